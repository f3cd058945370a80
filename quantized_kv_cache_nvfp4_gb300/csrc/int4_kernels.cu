// int4_kernels.cu -- INT4 affine codec encode kernels (plain pack and residual).
//
// Format ("vllm-rlt PR #166: INT4 KV packing/unpacking and cross-loop residual
// reconstruction", Purpose, and the review by 0z5a): groups of G values share an
// FP16 minimum and an FP16 scale; codes are computed in FP32 BEFORE the metadata is
// rounded to FP16; K groups run over G token rows per (head, channel), V groups over
// G channels per (token, head); the last group may be partial.  Per group, in order
// (binary32, nearest even):
//   mn = min x;  mx = max x;  sc = (mx - mn) / 15
//   code = 0 if sc == 0, else clamp(rint((x - mn) / sc), 0, 15)   (rint: ties even)
//   stored: fp16(mn), fp16(sc); two codes per byte, low nibble = even channel.
// Residual encode feeds the same codec with r = bf16(cur - prev) of the kept rows
// (same page, Purpose: residuals subtract the reconstructed predecessor in the
// input dtype; K groups follow the compact row order).
#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;

// Code of x in a group with FP32 minimum mn and scale sc > 0, rsc = RN(1 / sc):
// clamp(rint(RN(RN(x - mn) / sc)), 0, 15), usually without dividing.
//
// With d = RN(x - mn) >= 0, the estimate qe = RN(d * rsc) and the defined quotient
// q = RN(d / sc) both lie within 2 * 2^-24 (relative) of d / sc, and d / sc <= 15 *
// (1 + 2^-23) because x <= max; so after clamping to 15, |qe - q| < 2.9e-6 < 2^-17.
// When qe is more than 2^-17 away from the half-integers around it, q rounds to the
// same integer as qe (rint is ties-to-even, and no tie is possible there).
// Otherwise, and whenever sc is not a normal binary32 (rsc could overflow), the
// quotient is formed by the division itself.
//
// Rounding to an integer: for 0 <= v <= 15, RN(v + 1.5 * 2^23) has unit spacing, so
// it is v rounded to nearest with ties to even, and its low four mantissa bits are
// that integer.
constexpr float kRound = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ uint32_t int4_code(float x, float mn, float sc, float rsc) {
  const float d = __fsub_rn(x, mn);
  if (sc >= 0x1p-126f) {
    const float qe = fminf(__fmul_rn(d, rsc), 15.0f);
    const float t = __fadd_rn(qe, kRound);
    if (fabsf(__fsub_rn(qe, __fsub_rn(t, kRound))) < 0.49999237f)  // 0.5 - 2^-17
      return __float_as_uint(t) & 15u;
  }
  return __float_as_uint(__fadd_rn(fminf(__fdiv_rn(d, sc), 15.0f), kRound)) & 15u;
}

__device__ __forceinline__ float int4_rcp(float sc) { return sc != 0.0f ? __frcp_rn(sc) : 0.0f; }

// Codes of the two bf16 of w (lo, hi) -> one byte (lo | hi << 4), the same integers
// as int4_code (0 for a constant group, sc == 0).  The estimate, its rounding and its
// distance to the rounded integer are formed two at a time in f32x2.  No clamp is
// needed here: x <= max gives q <= 15 * (1 + 2^-22) < 15.5, which rounds to 15.
__device__ __forceinline__ uint32_t int4_pair(uint32_t w, float mnl, float mnh, float scl, float sch,
                                              float rscl, float rsch) {
  const uint64_t k2 = pack_f32x2(__float_as_uint(kRound), __float_as_uint(kRound));
  const uint64_t q2 = mul_f32x2(add_f32x2(pack_f32x2(w << 16, w & 0xFFFF0000u),
                                          pack_f32x2(__float_as_uint(-mnl), __float_as_uint(-mnh))),
                                pack_f32x2(__float_as_uint(rscl), __float_as_uint(rsch)));
  const uint64_t t2 = add_f32x2(q2, k2);
  uint32_t el, eh, tl, th;
  unpack_f32x2(sub_f32x2(q2, sub_f32x2(t2, k2)), el, eh);  // estimate - its rounded integer
  unpack_f32x2(t2, tl, th);
  const bool ok = fabsf(__uint_as_float(el)) < 0.49999237f && fabsf(__uint_as_float(eh)) < 0.49999237f &&
                  (scl >= 0x1p-126f || scl == 0.0f) && (sch >= 0x1p-126f || sch == 0.0f);
  if (ok) return (tl & 15u) | ((th & 15u) << 4);
  const uint32_t cl = scl != 0.0f ? int4_code(bf16lo(w), mnl, scl, rscl) : 0u;
  const uint32_t ch = sch != 0.0f ? int4_code(bf16hi(w), mnh, sch, rsch) : 0u;
  return cl | (ch << 4);
}

// The 8 bf16 values of one 16-byte chunk of a compact row (residual: bf16(cur-prev)).
// Returns false for a residual row whose position is out of range (values zero).
template <bool kResidual>
__device__ __forceinline__ bool load_chunk8(const Int4EncodeParams& p, int32_t row, int32_t h,
                                            int32_t col, uint32_t (&w)[4]) {
  int64_t src = row;
  if constexpr (kResidual) {
    if (p.pos != nullptr) src = LDX(p.pos + row);
    if (src < 0 || src >= p.src_rows) {
      w[0] = w[1] = w[2] = w[3] = 0u;
      return false;
    }
  }
  load16B(p.x + src * p.row_pitch + static_cast<int64_t>(h) * p.head_pitch + col, w);
  if constexpr (kResidual) {
    uint32_t q[4];
    load16B(p.prev + src * p.prev_row_pitch + static_cast<int64_t>(h) * p.prev_head_pitch + col, q);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = pack_bf16x2(__fsub_rn(bf16lo(w[i]), bf16lo(q[i])),
                         __fsub_rn(bf16hi(w[i]), bf16hi(q[i])));
  }
  return true;
}

template <bool kResidual>
__device__ __forceinline__ void check_pos(const Int4EncodeParams& p, int32_t row) {
  if constexpr (kResidual) {
    if (p.pos == nullptr) return;
    const int32_t ps = LDX(p.pos + row);
    bool bad = ps < 0 || ps >= p.src_rows;
    if (row > 0 && LDX(p.pos + row - 1) >= ps) bad = true;
    if (bad) set_status(p.status, 4u);
    if (p.pos_out != nullptr) STX(p.pos_out + row, ps);
  }
}

// KEY kind: a column task is (group of G rows, head, 8-channel chunk).  RS = G / RPL
// lanes share a task; each holds its RPL rows of the chunk in registers (all loads
// issued together), so every row is read once.  The RS partial minima/maxima meet in
// a xor butterfly, then each lane codes its own rows.  A warp holds 32/RS
// consecutive chunks of a row, so each row read is one coalesced span per row split.
template <bool kResidual, int RS, int RPL>
__global__ void __launch_bounds__(kThreads) int4_key_kernel(const Int4EncodeParams p) {
  constexpr int CW = 32 / RS;
  const int lane = threadIdx.x & 31;
  const int rs = lane / CW;
  const int cl = lane % CW;
  const int32_t nchunk = p.D / 8;
  const int32_t ngroups = (p.rows + p.G - 1) / p.G;
  const int64_t ntask = static_cast<int64_t>(ngroups) * p.H * nchunk;
  const int64_t nwtask = (ntask + CW - 1) / CW;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t wt = blockIdx.x * static_cast<int64_t>(kThreads / 32) + threadIdx.x / 32; wt < nwtask;
       wt += nwarps) {
    const int64_t task = wt * CW + cl;
    const bool valid = task < ntask;
    const int64_t tk = valid ? task : 0;
    const int32_t chunk = static_cast<int32_t>(tk % nchunk);
    const int32_t h = static_cast<int32_t>((tk / nchunk) % p.H);
    const int32_t g = static_cast<int32_t>(tk / (static_cast<int64_t>(nchunk) * p.H));
    const int32_t r0 = g * p.G;
    const int32_t r1 = valid ? min(p.rows, r0 + p.G) : r0;
    const int32_t col = chunk * 8;

    uint32_t v[RPL][4];
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int32_t r = r0 + rs + k * RS;
      if (r < r1) {
        load_chunk8<kResidual>(p, r, h, col, v[k]);
      } else {
        v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0u;
      }
    }
    // group minimum / maximum per channel, in the bf16 order keys (-0 below +0)
    uint32_t kmn[4], kmx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kmn[i] = 0xFFFFFFFFu;
      kmx[i] = 0u;
    }
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      if (r0 + rs + k * RS >= r1) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t key = bf16x2_key(v[k][i]);
        kmn[i] = min_u16x2(kmn[i], key);
        kmx[i] = max_u16x2(kmx[i], key);
      }
    }
#pragma unroll
    for (int o = CW; o < 32; o <<= 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kmn[i] = min_u16x2(kmn[i], __shfl_xor_sync(0xFFFFFFFFu, kmn[i], o));
        kmx[i] = max_u16x2(kmx[i], __shfl_xor_sync(0xFFFFFFFFu, kmx[i], o));
      }
    }
    float mn[8], mx[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a = bf16x2_unkey(kmn[i]), b = bf16x2_unkey(kmx[i]);
      mn[2 * i] = bf16lo(a);
      mn[2 * i + 1] = bf16hi(a);
      mx[2 * i] = bf16lo(b);
      mx[2 * i + 1] = bf16hi(b);
    }
    if (!valid) continue;
    float sc[8], rsc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sc[i] = __fdiv_rn(__fsub_rn(mx[i], mn[i]), 15.0f);
      rsc[i] = int4_rcp(sc[i]);
    }
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int32_t r = r0 + rs + k * RS;
      if (r >= r1) continue;
      if (chunk == 0 && h == 0) check_pos<kResidual>(p, r);
      uint32_t packed = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        packed |= int4_pair(v[k][i], mn[2 * i], mn[2 * i + 1], sc[2 * i], sc[2 * i + 1], rsc[2 * i],
                            rsc[2 * i + 1])
                  << (8 * i);
      STX(reinterpret_cast<uint32_t*>(p.dst.codes + (static_cast<int64_t>(r) * p.H + h) * (p.D / 2) +
                                      col / 2),
          packed);
    }
    if (rs == 0) {
      uint32_t m16[4], s16[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m16[i] = static_cast<uint32_t>(f32_to_f16_bits(mn[2 * i])) |
                 (static_cast<uint32_t>(f32_to_f16_bits(mn[2 * i + 1])) << 16);
        s16[i] = static_cast<uint32_t>(f32_to_f16_bits(sc[2 * i])) |
                 (static_cast<uint32_t>(f32_to_f16_bits(sc[2 * i + 1])) << 16);
      }
      const int64_t m = (static_cast<int64_t>(g) * p.H + h) * p.D + col;
      store16B(p.dst.mn + m, m16);
      store16B(p.dst.sc + m, s16);
    }
  }
}

// KEY kind, tiled through shared memory: a block takes one tile (a group of up to G
// rows x the D channels of one head) at a time, in kStages shared-memory buffers.
//  1. the tile's rows are copied into shared memory with 16-byte cp.async copies,
//     all issued at once (consecutive threads, consecutive chunks of a row); with two
//     stages the next tile's copies are in flight while this tile is coded.  Residual
//     mode gathers the rows at pos[] from cur and prev into two planes;
//  2. thread (rq, cp) takes channel pair cp over rows rq, rq + RQ, ... (RQ = 512 / D
//     row splits; a warp reads consecutive words: no bank conflicts), forms the
//     residual bf16(cur - prev) in place, and leaves its partial minimum/maximum in
//     shared memory; after a barrier every thread combines the RQ partials of its
//     pair, so the group's FP32 minimum and scale are known;
//  3. each thread codes its rows of the pair (one byte per row, a warp writes 32
//     consecutive bytes) and the rq == 0 threads write the FP16 metadata.
template <bool kResidual, int kStages>
__global__ void __launch_bounds__(kThreads) int4_key_tile_kernel(const Int4EncodeParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int kPlanes = kResidual ? 2 : 1;
  const int D = p.D;
  const int nchunk = D / 8;     // 16-byte chunks per row
  const int npair = D / 2;      // channel pairs = 32-bit words per row
  const int RQ = kThreads / npair;
  const int tid = threadIdx.x;
  const int cp = tid % npair;
  const int rq = tid / npair;
  const int tile_words = p.G * npair;
  uint32_t* const buf = reinterpret_cast<uint32_t*>(smem);  // [kStages][kPlanes][G][D/2]
  uint32_t* const part = buf + kStages * kPlanes * tile_words;  // [2][RQ][D/2] keys
  const int32_t ngroups = (p.rows + p.G - 1) / p.G;
  const int64_t ntiles = static_cast<int64_t>(ngroups) * p.H;

  // copies of tile `tile_id` into stage `st` (nothing past the last tile)
  auto issue = [&](int64_t tile_id, int st) {
    if (tile_id >= ntiles) return;
    const int32_t g = static_cast<int32_t>(tile_id / p.H);
    const int32_t h = static_cast<int32_t>(tile_id % p.H);
    const int32_t r0 = g * p.G;
    const int32_t nr = min(p.G, p.rows - r0);
    uint32_t* const cur = buf + st * kPlanes * tile_words;
    for (int c = tid; c < nr * nchunk; c += kThreads) {
      const int row = c / nchunk;
      const int col = (c % nchunk) * 8;
      uint32_t* const dst = cur + row * npair + col / 2;
      int64_t src = r0 + row;
      if constexpr (kResidual) {
        if (p.pos != nullptr) src = LDX(p.pos + r0 + row);
        if (src < 0 || src >= p.src_rows) {  // a bad position codes zeros (and is flagged)
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(dst + tile_words) = make_uint4(0u, 0u, 0u, 0u);
          continue;
        }
        cp_async16(dst + tile_words,
                   p.prev + src * p.prev_row_pitch + static_cast<int64_t>(h) * p.prev_head_pitch + col);
      }
      cp_async16(dst, p.x + src * p.row_pitch + static_cast<int64_t>(h) * p.head_pitch + col);
    }
  };

  int64_t tile_id = blockIdx.x;
  issue(tile_id, 0);
  cp_async_commit();
  if constexpr (kStages == 2) {
    issue(tile_id + gridDim.x, 1);
    cp_async_commit();
  }
  for (int it = 0; tile_id < ntiles; tile_id += gridDim.x, ++it) {
    const int st = kStages == 2 ? (it & 1) : 0;
    if constexpr (kStages == 2) {
      cp_async_wait<1>();  // this tile's group is complete; the next may be in flight
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int32_t g = static_cast<int32_t>(tile_id / p.H);
    const int32_t h = static_cast<int32_t>(tile_id % p.H);
    const int32_t r0 = g * p.G;
    const int32_t nr = min(p.G, p.rows - r0);
    uint32_t* const tile = buf + st * kPlanes * tile_words;
    // 2. column minimum and maximum of the pair in bf16 order keys (-0 below +0;
    //    residual: the difference is formed first)
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
    if (rq < RQ) {
      for (int row = rq; row < nr; row += RQ) {
        uint32_t v = tile[row * npair + cp];
        if constexpr (kResidual) {
          const uint32_t q = tile[tile_words + row * npair + cp];
          v = pack_bf16x2(__fsub_rn(bf16lo(v), bf16lo(q)), __fsub_rn(bf16hi(v), bf16hi(q)));
          tile[row * npair + cp] = v;  // read back by this same thread in step 3
        }
        const uint32_t key = bf16x2_key(v);
        kmn = min_u16x2(kmn, key);
        kmx = max_u16x2(kmx, key);
      }
      part[rq * npair + cp] = kmn;
      part[(RQ + rq) * npair + cp] = kmx;
    }
    __syncthreads();
    if (rq < RQ) {
      for (int k = 0; k < RQ; ++k) {
        kmn = min_u16x2(kmn, part[k * npair + cp]);
        kmx = max_u16x2(kmx, part[(RQ + k) * npair + cp]);
      }
      const uint32_t wmn = bf16x2_unkey(kmn), wmx = bf16x2_unkey(kmx);
      const float mnl = bf16lo(wmn), mnh = bf16hi(wmn), mxl = bf16lo(wmx), mxh = bf16hi(wmx);
      const float scl = __fdiv_rn(__fsub_rn(mxl, mnl), 15.0f);
      const float sch = __fdiv_rn(__fsub_rn(mxh, mnh), 15.0f);
      const float rsl = int4_rcp(scl), rsh = int4_rcp(sch);
      // 3. codes of this thread's rows
      for (int row = rq; row < nr; row += RQ) {
        if (cp == 0 && h == 0) check_pos<kResidual>(p, r0 + row);
        const uint32_t byte = int4_pair(tile[row * npair + cp], mnl, mnh, scl, sch, rsl, rsh);
        STX(p.dst.codes + (static_cast<int64_t>(r0 + row) * p.H + h) * npair + cp, static_cast<uint8_t>(byte));
      }
      if (rq == 0) {
        const int64_t m = (static_cast<int64_t>(g) * p.H + h) * D + 2 * cp;
        STX(reinterpret_cast<uint32_t*>(p.dst.mn + m),
            static_cast<uint32_t>(f32_to_f16_bits(mnl)) | (static_cast<uint32_t>(f32_to_f16_bits(mnh)) << 16));
        STX(reinterpret_cast<uint32_t*>(p.dst.sc + m),
            static_cast<uint32_t>(f32_to_f16_bits(scl)) | (static_cast<uint32_t>(f32_to_f16_bits(sch)) << 16));
      }
    }
    __syncthreads();  // stage st and the partials are free again
    issue(tile_id + static_cast<int64_t>(kStages) * gridDim.x, st);
    cp_async_commit();
  }
  cp_async_wait<0>();  // only empty groups remain; nothing is left in flight at exit
}

// VALUE kind: one lane per 16-channel block of a row; a group spans W = min(G/16, L)
// aligned lanes, reduced with a xor butterfly of uniform width.
template <int L, bool kResidual>
__global__ void __launch_bounds__(kThreads) int4_value_kernel(const Int4EncodeParams p) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int b = lane % L;
  const int sub = lane / L;
  const int nb = p.D / 16;
  const int W = min(p.G / 16, L);
  const int ngv = (p.D + p.G - 1) / p.G;
  const uint32_t total = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H);
  const uint32_t stride = gridDim.x * (kThreads / 32) * kRowsPerWarp;
  const bool has = b < nb;

  // the 16 values of this lane's block of row `rw` (zeros when there is none)
  auto load_row = [&](uint32_t rw, uint32_t (&w)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0u;
    if (rw >= total || !has) return;
    uint32_t ru, hu;
    p.div_h.divmod(rw, ru, hu);
    uint32_t a[4], c[4];
    load_chunk8<kResidual>(p, static_cast<int32_t>(ru), static_cast<int32_t>(hu), 16 * b, a);
    load_chunk8<kResidual>(p, static_cast<int32_t>(ru), static_cast<int32_t>(hu), 16 * b + 8, c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = a[i];
      w[4 + i] = c[i];
    }
  };

  uint32_t row = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
  uint32_t w[8];
  load_row(row, w);
  for (; row - sub < total; row += stride) {
    const bool valid = row < total && has;
    uint32_t ru, hu;
    p.div_h.divmod(valid ? row : 0u, ru, hu);
    const int32_t r = static_cast<int32_t>(ru), h = static_cast<int32_t>(hu);
    uint32_t nw[8];
    load_row(row + stride, nw);  // the next row's loads before this row's arithmetic
    if (valid && b == 0 && h == 0) check_pos<kResidual>(p, r);
    // the group's minimum and maximum in bf16 order keys (-0 below +0); one word
    // carries the minimum key (low half) and the complemented maximum key (high half),
    // so a single unsigned min per butterfly round reduces both
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
    if (valid) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t key = bf16x2_key(w[i]);
        kmn = min_u16x2(kmn, key);
        kmx = max_u16x2(kmx, key);
      }
    }
    kmn = min_u16x2(kmn, __byte_perm(kmn, 0u, 0x1032));  // both halves: the lane minimum
    kmx = max_u16x2(kmx, __byte_perm(kmx, 0u, 0x1032));
    uint32_t mm = (kmn & 0xFFFFu) | (~kmx << 16);
    for (int o = 1; o < W; o <<= 1)  // W is uniform: every lane runs the same shuffles
      mm = min_u16x2(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, o));
    if (!valid) {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = nw[i];
      continue;
    }
    const uint32_t mnmx = bf16x2_unkey(mm ^ 0xFFFF0000u);  // low: minimum, high: maximum
    const float lmn = bf16lo(mnmx), lmx = bf16hi(mnmx);
    const float sc = __fdiv_rn(__fsub_rn(lmx, lmn), 15.0f);
    const float rsc = int4_rcp(sc);
    uint32_t c0 = 0u, c1 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = int4_pair(w[i], lmn, lmn, sc, sc, rsc, rsc);
      if (i < 4)
        c0 |= byte << (8 * i);
      else
        c1 |= byte << (8 * (i - 4));
    }
    const int64_t drow = static_cast<int64_t>(r) * p.H + h;
    store8B(p.dst.codes + drow * (p.D / 2) + 8 * b, c0, c1);
    if ((16 * b) % p.G == 0) {
      const int64_t m = drow * ngv + (16 * b) / p.G;
      STX(p.dst.mn + m, f32_to_f16_bits(lmn));
      STX(p.dst.sc + m, f32_to_f16_bits(sc));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = nw[i];
  }
}

template <typename K>
int grid_cap(K kernel, int64_t work_items, int items_per_cta) {
  int occ = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0);
  if (occ < 1) occ = 1;
  int64_t need = (work_items + items_per_cta - 1) / items_per_cta;
  int64_t cap = static_cast<int64_t>(num_sms()) * occ;
  if (need < 1) need = 1;
  return static_cast<int>(need < cap ? need : cap);
}

template <int L, bool kRes>
cudaError_t value_launch(const Int4EncodeParams& p, cudaStream_t s) {
  auto k = int4_value_kernel<L, kRes>;
  int grid = grid_cap(k, static_cast<int64_t>(p.rows) * p.H, (kThreads / 32) * (32 / L));
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("int4_value_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

template <bool kRes>
cudaError_t value_dispatch(const Int4EncodeParams& p, cudaStream_t s) {
  int nb = p.D / 16, L = 1;
  while (L < nb) L <<= 1;
  switch (L) {
    case 1: return value_launch<1, kRes>(p, s);
    case 2: return value_launch<2, kRes>(p, s);
    case 4: return value_launch<4, kRes>(p, s);
    case 8: return value_launch<8, kRes>(p, s);
    case 16: return value_launch<16, kRes>(p, s);
    case 32: return value_launch<32, kRes>(p, s);
  }
  return cudaErrorInvalidValue;
}

template <bool kRes, int RS, int RPL>
cudaError_t key_launch(const Int4EncodeParams& p, int64_t ntask, cudaStream_t s) {
  auto k = int4_key_kernel<kRes, RS, RPL>;
  const int64_t warps = (ntask + 32 / RS - 1) / (32 / RS);
  const int grid = grid_cap(k, warps, kThreads / 32);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("int4_key_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

// Shared memory of the tile kernel: kStages x planes tiles of G x D bf16, plus the
// [2][RQ][D/2] partial key words.
size_t key_tile_smem(int G, int D, int stages, int planes) {
  return static_cast<size_t>(stages) * planes * G * D * 2 + 2 * static_cast<size_t>(kThreads / (D / 2)) * D * 2;
}

constexpr size_t kTileSmemCap = 110 * 1024;  // two blocks per SM at least

template <bool kRes, int kStages>
cudaError_t key_tile_launch(const Int4EncodeParams& p, cudaStream_t s) {
  auto k = int4_key_tile_kernel<kRes, kStages>;
  const size_t smem = key_tile_smem(p.G, p.D, kStages, kRes ? 2 : 1);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  int occ = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, smem);
  if (occ < 1) occ = 1;
  const int64_t tiles = static_cast<int64_t>((p.rows + p.G - 1) / p.G) * p.H;
  const int64_t cap = static_cast<int64_t>(num_sms()) * occ;
  const int grid = static_cast<int>(tiles < cap ? (tiles < 1 ? 1 : tiles) : cap);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("int4_key_tile_kernel", s, k<<<grid, kThreads, smem, s>>>(p); e = cudaGetLastError());
  return e;
}

template <bool kRes>
cudaError_t key_dispatch(const Int4EncodeParams& p, cudaStream_t s) {
  const int planes = kRes ? 2 : 1;
  if (p.D >= 16 && key_tile_smem(p.G, p.D, 2, planes) <= kTileSmemCap) return key_tile_launch<kRes, 2>(p, s);
  if (p.D >= 16 && key_tile_smem(p.G, p.D, 1, planes) <= kTileSmemCap) return key_tile_launch<kRes, 1>(p, s);
  const int64_t ntask = static_cast<int64_t>((p.rows + p.G - 1) / p.G) * p.H * (p.D / 8);
  switch (p.G) {  // RS = G / RPL lanes per column task
    case 16: return key_launch<kRes, 2, 8>(p, ntask, s);
    case 32: return key_launch<kRes, 4, 8>(p, ntask, s);
    case 64: return key_launch<kRes, 8, 8>(p, ntask, s);
    case 128: return key_launch<kRes, 16, 8>(p, ntask, s);
    case 256: return key_launch<kRes, 32, 8>(p, ntask, s);
    case 512: return key_launch<kRes, 32, 16>(p, ntask, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_int4_encode(const Int4EncodeParams& p, cudaStream_t s) {
  if (p.kind == 0) return p.residual ? key_dispatch<true>(p, s) : key_dispatch<false>(p, s);
  return p.residual ? value_dispatch<true>(p, s) : value_dispatch<false>(p, s);
}

}  // namespace kvq
