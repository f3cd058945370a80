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
// The minimum and maximum order -0 below +0 (IEEE 754-2019 minimum/maximum).
// Residual encode feeds the same codec with r = bf16(cur - prev) of the kept rows
// (same page, Purpose: residuals subtract the reconstructed predecessor in the
// input dtype; K groups follow the compact row order).
#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;

// Quotients without dividing.  Both divisions of the format are formed from a
// correctly rounded reciprocal y = RN(1/b) and FMA residuals (Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev.
// 34(1), 1990: when q is within one ulp of a/b and y = RN(1/b), the residual
// a - b*q is exact and RN(q + (a - b*q)*y) = RN(a/b), barring underflow).
//
// Group scale: sc = RN(D / 15) for D = RN(mx - mn).  q0 = RN(D * RN(1/15)) plus one
// residual step equals the IEEE quotient for every binary32 D in [2^-64, FLT_MAX]
// (checked for all of them, 1.6e9 values); smaller D divide.
constexpr float kRcp15 = 0x1.111112p-4f;  // RN(1/15)

__device__ __forceinline__ float int4_scale(float D) {
  if (D >= 0x1p-64f && D <= 3.4028235e38f) {
    const float q0 = __fmul_rn(D, kRcp15);
    return __fmaf_rn(__fmaf_rn(-q0, 15.0f, D), kRcp15, q0);
  }
  return __fdiv_rn(D, 15.0f);
}

// Element quotient q = RN(d / sc), d = RN(x - mn) >= 0, for a scale sc >= 2^-64 with
// y = RN(1/sc): q0 = RN(d*y) is within 2u + u^2 of d/sc (u = 2^-24); one residual
// step leaves a relative error below 4u^2, so q1 is within one ulp and a second step
// returns RN(d/sc) by the theorem above.  The second residual is exact while
// e(sc) + e(q) >= -103 (binary exponents), i.e. for every q >= 2^-39 here; a smaller
// q codes 0 either way (every step stays far below 0.5).  Scales under 2^-64 divide.
// A constant group (sc = 0, so d = 0) uses y = 0, which gives q = 0.
__device__ __forceinline__ bool int4_fast_scale(float sc) { return sc >= 0x1p-64f || sc == 0.0f; }
__device__ __forceinline__ float int4_recip(float sc) { return sc != 0.0f ? __frcp_rn(sc) : 0.0f; }

// Rounding to an integer: for 0 <= q < 15.5, RN(q + 1.5 * 2^23) has unit spacing, so
// it is q rounded to nearest with ties to even, and its low four mantissa bits are
// that integer.  q <= D / sc <= 15 / (1 - 2^-24) < 15.5 (d <= D), so no clamp applies.
constexpr float kRound = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t dup_f32x2(float v) {
  return pack_f32x2(__float_as_uint(v), __float_as_uint(v));
}
// (x_lo + c_lo, x_hi + c_hi) in binary32 for the two bf16 of w and the pair c, each sum
// rounded once (the bf16 -> f32 widening is exact): mixed-precision adds.
__device__ __forceinline__ uint64_t add_bf16x2_f32x2(uint32_t w, uint64_t c) {
  uint32_t cl, ch;
  unpack_f32x2(c, cl, ch);
  float dl, dh;
  asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %4;\n\t}"
      : "=f"(dl), "=f"(dh)
      : "r"(w), "f"(__uint_as_float(cl)), "f"(__uint_as_float(ch)));
  return pack_f32x2(__float_as_uint(dl), __float_as_uint(dh));
}

// Codes of the 8 bf16 of words w[0..3] (channel 2i in the low half of w[i], 2i + 1 in
// the high half) for fast scales, with per-channel-pair parameters as f32x2 pairs:
// nmn = -minimum, nsc = -scale, y = RN(1/scale).  Byte i of the result holds w[i]'s
// two codes, low nibble = even channel.  With t = K + n (n <= 15) the float bits end in
// n, so t_hi * 16 + t_lo carries nothing out of its low byte, which is n_lo | n_hi << 4.
__device__ __forceinline__ uint32_t int4_codes8(const uint32_t (&w)[4], const uint64_t (&nmn)[4],
                                                const uint64_t (&nsc)[4], const uint64_t (&y)[4]) {
  const uint64_t k2 = dup_f32x2(kRound);
  uint32_t byte[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t d = add_bf16x2_f32x2(w[i], nmn[i]);
    const uint64_t q0 = mul_f32x2(d, y[i]);
    const uint64_t q1 = fma_f32x2(fma_f32x2(q0, nsc[i], d), y[i], q0);
    const uint64_t q2 = fma_f32x2(fma_f32x2(q1, nsc[i], d), y[i], q1);
    uint32_t tl, th;
    unpack_f32x2(add_f32x2(q2, k2), tl, th);
    byte[i] = th * 16u + tl;
  }
  return __byte_perm(__byte_perm(byte[0], byte[1], 0x0040u), __byte_perm(byte[2], byte[3], 0x0040u), 0x5410u);
}

// The same codes by division, element by element (the defined arithmetic), for chunks
// holding a scale below 2^-64; same parameters.
__device__ __forceinline__ uint32_t int4_codes8_div(const uint32_t (&w)[4], const uint64_t (&nmn)[4],
                                                    const uint64_t (&nsc)[4]) {
  uint32_t out = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t ml, mh, sl, sh;
    unpack_f32x2(nmn[i], ml, mh);
    unpack_f32x2(nsc[i], sl, sh);
    const float x[2] = {bf16lo(w[i]), bf16hi(w[i])};
    const float m[2] = {-__uint_as_float(ml), -__uint_as_float(mh)};
    const float s[2] = {-__uint_as_float(sl), -__uint_as_float(sh)};
    uint32_t c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      c[j] = s[j] != 0.0f
                 ? __float_as_uint(__fadd_rn(fminf(__fdiv_rn(__fsub_rn(x[j], m[j]), s[j]), 15.0f), kRound)) & 15u
                 : 0u;
    out |= (c[0] | (c[1] << 4)) << (8 * i);
  }
  return out;
}

// Group minimum and maximum of packed bf16 words: min/max.bf16x2 (a minimum or
// maximum of bf16 values is one of them, so nothing rounds) and the OR of the words.
// The hardware may return either zero for a (-0, +0) pair; only the sign of a zero
// MINIMUM is stored, and a zero minimum means no element is negative, so the group
// holds a -0 exactly when a sign bit is set in the OR.  (The sign of a zero maximum
// never matters: sc = mx - mn is +0 either way.)
__device__ __forceinline__ uint32_t hmin2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// A group minimum in FP32 from its bf16 bits (low 16 bits of m) and the group's OR of
// sign bits (nonzero when some element has its sign bit set).
__device__ __forceinline__ float group_min(uint32_t m, uint32_t any_sign) {
  const float v = __uint_as_float(m << 16);
  return v == 0.0f ? __uint_as_float(any_sign != 0u ? 0x80000000u : 0u) : v;
}
constexpr uint32_t kPosInf2 = 0x7F807F80u;  // bf16x2 +inf, +inf
constexpr uint32_t kNegInf2 = 0xFF80FF80u;  // bf16x2 -inf, -inf

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

// KEY kind, register fallback for tiles too large for shared memory: a column task is
// (group of G rows, head, 8-channel chunk).  RS = G / RPL lanes share a task; each
// holds its RPL rows of the chunk in registers (all loads issued together), so every
// row is read once.  The RS partial minima/maxima meet in a xor butterfly (in bf16
// order keys, -0 below +0), then each lane codes its own rows.
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
    if (!valid) continue;
    float mn[8], sc[8];
    uint64_t nmn[4], nsc[4], y[4];
    bool fast = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a = bf16x2_unkey(kmn[i]), b = bf16x2_unkey(kmx[i]);
      mn[2 * i] = bf16lo(a);
      mn[2 * i + 1] = bf16hi(a);
      sc[2 * i] = int4_scale(__fsub_rn(bf16lo(b), mn[2 * i]));
      sc[2 * i + 1] = int4_scale(__fsub_rn(bf16hi(b), mn[2 * i + 1]));
      nmn[i] = pack_f32x2(__float_as_uint(-mn[2 * i]), __float_as_uint(-mn[2 * i + 1]));
      nsc[i] = pack_f32x2(__float_as_uint(-sc[2 * i]), __float_as_uint(-sc[2 * i + 1]));
      y[i] = pack_f32x2(__float_as_uint(int4_recip(sc[2 * i])), __float_as_uint(int4_recip(sc[2 * i + 1])));
      fast = fast && int4_fast_scale(sc[2 * i]) && int4_fast_scale(sc[2 * i + 1]);
    }
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int32_t r = r0 + rs + k * RS;
      if (r >= r1) continue;
      if (chunk == 0 && h == 0) check_pos<kResidual>(p, r);
      STX(reinterpret_cast<uint32_t*>(p.dst.codes + (static_cast<int64_t>(r) * p.H + h) * (p.D / 2) + col / 2),
          fast ? int4_codes8(v[k], nmn, nsc, y) : int4_codes8_div(v[k], nmn, nsc));
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
// Thread (rq, ch) owns 16-byte chunk ch (channels 8ch .. 8ch + 7) of rows rq,
// rq + RP, ... (RP = 256 / (D / 8) rows per pass) through every step:
//  1. the tile's rows are copied into shared memory with 16-byte cp.async copies; with
//     two stages the next tile's copies are in flight while this tile is coded.
//     Residual mode gathers the rows at pos[] from cur and prev into two planes;
//  2. each thread reduces its rows of its chunk (residual: forms bf16(cur - prev) in
//     place first) to partial min / max / sign-OR words;
//  3. one thread per channel pair combines the RP partials, computes the group's
//     minimum, scale and reciprocal, keeps them in shared memory and writes the FP16
//     metadata;
//  4. each thread codes its rows of its chunk: 8 codes -> one 32-bit store.
template <bool kResidual, int kStages>
__global__ void __launch_bounds__(kThreads) int4_key_tile_kernel(const Int4EncodeParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int kPlanes = kResidual ? 2 : 1;
  const int D = p.D;
  const int nchunk = D / 8;  // 16-byte chunks per row
  const int npair = D / 2;   // 32-bit words per row
  const int RP = kThreads / nchunk;
  const int tid = threadIdx.x;
  const bool worker = tid < RP * nchunk;
  const int ch = tid % nchunk;
  const int rq = tid / nchunk;
  const int tile_words = p.G * npair;
  uint32_t* const buf = reinterpret_cast<uint32_t*>(smem);                             // [kStages][kPlanes][G][D/2]
  uint4* const part = reinterpret_cast<uint4*>(buf + kStages * kPlanes * tile_words);  // [3][RP][D/8]
  float2* const prm = reinterpret_cast<float2*>(part + 3 * RP * nchunk);               // [3][D/2]
  const uint32_t ntiles = static_cast<uint32_t>((p.rows + p.G - 1) / p.G) * static_cast<uint32_t>(p.H);

  // copies of tile `tile` into stage `st` (nothing past the last tile)
  auto issue = [&](uint32_t tile, int st) {
    if (!worker || tile >= ntiles) return;
    uint32_t g, h;
    p.div_h.divmod(tile, g, h);
    const int32_t r0 = static_cast<int32_t>(g) * p.G;
    const int32_t nr = min(p.G, p.rows - r0);
    uint32_t* const cur = buf + st * kPlanes * tile_words + ch * 4;
    for (int row = rq; row < nr; row += RP) {
      uint32_t* const dst = cur + row * npair;
      int64_t src = r0 + row;
      if constexpr (kResidual) {
        if (p.pos != nullptr) src = LDX(p.pos + r0 + row);
        if (src < 0 || src >= p.src_rows) {  // a bad position codes zeros (and is flagged)
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(dst + tile_words) = make_uint4(0u, 0u, 0u, 0u);
          continue;
        }
        cp_async16(dst + tile_words,
                   p.prev + src * p.prev_row_pitch + static_cast<int64_t>(h) * p.prev_head_pitch + ch * 8);
      }
      cp_async16(dst, p.x + src * p.row_pitch + static_cast<int64_t>(h) * p.head_pitch + ch * 8);
    }
  };

  uint32_t tile = blockIdx.x;
  issue(tile, 0);
  cp_async_commit();
  if constexpr (kStages == 2) {
    issue(tile + gridDim.x, 1);
    cp_async_commit();
  }
  for (int it = 0; tile < ntiles; tile += gridDim.x, ++it) {
    const int st = kStages == 2 ? (it & 1) : 0;
    if constexpr (kStages == 2) {
      cp_async_wait<1>();  // this tile's group is complete; the next may be in flight
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    uint32_t g, h;
    p.div_h.divmod(tile, g, h);
    const int32_t r0 = static_cast<int32_t>(g) * p.G;
    const int32_t nr = min(p.G, p.rows - r0);
    uint32_t* const tw = buf + st * kPlanes * tile_words + ch * 4;  // this thread's column
    // 2. partial minimum / maximum / sign-OR of this thread's rows of its chunk
    if (worker) {
      uint32_t mn[4] = {kPosInf2, kPosInf2, kPosInf2, kPosInf2};
      uint32_t mx[4] = {kNegInf2, kNegInf2, kNegInf2, kNegInf2};
      uint32_t sg[4] = {0u, 0u, 0u, 0u};
      for (int row = rq; row < nr; row += RP) {
        uint4 v = *reinterpret_cast<const uint4*>(tw + row * npair);
        if constexpr (kResidual) {
          const uint4 q = *reinterpret_cast<const uint4*>(tw + tile_words + row * npair);
          v.x = pack_bf16x2(__fsub_rn(bf16lo(v.x), bf16lo(q.x)), __fsub_rn(bf16hi(v.x), bf16hi(q.x)));
          v.y = pack_bf16x2(__fsub_rn(bf16lo(v.y), bf16lo(q.y)), __fsub_rn(bf16hi(v.y), bf16hi(q.y)));
          v.z = pack_bf16x2(__fsub_rn(bf16lo(v.z), bf16lo(q.z)), __fsub_rn(bf16hi(v.z), bf16hi(q.z)));
          v.w = pack_bf16x2(__fsub_rn(bf16lo(v.w), bf16lo(q.w)), __fsub_rn(bf16hi(v.w), bf16hi(q.w)));
          *reinterpret_cast<uint4*>(tw + row * npair) = v;  // read back by this thread in step 4
        }
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mn[i] = hmin2(mn[i], w[i]);
          mx[i] = hmax2(mx[i], w[i]);
          sg[i] |= w[i];
        }
      }
      part[(0 * RP + rq) * nchunk + ch] = make_uint4(mn[0], mn[1], mn[2], mn[3]);
      part[(1 * RP + rq) * nchunk + ch] = make_uint4(mx[0], mx[1], mx[2], mx[3]);
      part[(2 * RP + rq) * nchunk + ch] = make_uint4(sg[0], sg[1], sg[2], sg[3]);
    }
    __syncthreads();
    // 3. per channel pair (32-bit word w = tid): the group's minimum, scale and
    //    reciprocal, kept in shared memory (minimum and scale negated) at
    //    [param][w % 4][w / 4] (so step 4 reads consecutive words), and the FP16 metadata
    if (tid < npair) {
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(part);  // [3][RP][D/2] words
      uint32_t m = kPosInf2, M = kNegInf2, sgn = 0u;
      for (int k = 0; k < RP; ++k) {
        m = hmin2(m, pw[(0 * RP + k) * npair + tid]);
        M = hmax2(M, pw[(1 * RP + k) * npair + tid]);
        sgn |= pw[(2 * RP + k) * npair + tid];
      }
      const float mnl = group_min(m, sgn & 0x8000u), mnh = group_min(m >> 16, sgn & 0x80000000u);
      const float scl = int4_scale(__fsub_rn(bf16lo(M), mnl));
      const float sch = int4_scale(__fsub_rn(bf16hi(M), mnh));
      const int slot = (tid % 4) * nchunk + tid / 4;
      prm[slot] = make_float2(-mnl, -mnh);
      prm[4 * nchunk + slot] = make_float2(-scl, -sch);
      prm[8 * nchunk + slot] = make_float2(int4_recip(scl), int4_recip(sch));
      const int64_t mi = (static_cast<int64_t>(g) * p.H + h) * D + 2 * tid;
      STX(reinterpret_cast<uint32_t*>(p.dst.mn + mi),
          static_cast<uint32_t>(f32_to_f16_bits(mnl)) | (static_cast<uint32_t>(f32_to_f16_bits(mnh)) << 16));
      STX(reinterpret_cast<uint32_t*>(p.dst.sc + mi),
          static_cast<uint32_t>(f32_to_f16_bits(scl)) | (static_cast<uint32_t>(f32_to_f16_bits(sch)) << 16));
    }
    __syncthreads();
    // 4. codes of this thread's rows of its chunk
    if (worker) {
      const uint64_t* const pq = reinterpret_cast<const uint64_t*>(prm);
      uint64_t nmn[4], nsc[4], y[4];
      bool fast = true;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        nmn[i] = pq[i * nchunk + ch];
        nsc[i] = pq[(4 + i) * nchunk + ch];
        y[i] = pq[(8 + i) * nchunk + ch];
        uint32_t sl, sh;
        unpack_f32x2(nsc[i], sl, sh);
        fast = fast && int4_fast_scale(-__uint_as_float(sl)) && int4_fast_scale(-__uint_as_float(sh));
      }
      uint8_t* const cbase = p.dst.codes + static_cast<int64_t>(h) * npair + ch * 4;
      const int64_t cstride = static_cast<int64_t>(p.H) * npair;
      for (int row = rq; row < nr; row += RP) {
        if (ch == 0 && h == 0) check_pos<kResidual>(p, r0 + row);
        const uint4 v = *reinterpret_cast<const uint4*>(tw + row * npair);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        STX(reinterpret_cast<uint32_t*>(cbase + (r0 + row) * cstride),
            fast ? int4_codes8(w, nmn, nsc, y) : int4_codes8_div(w, nmn, nsc));
      }
    }
    __syncthreads();  // stage st, the partials and the parameters are free again
    issue(tile + static_cast<uint32_t>(kStages) * gridDim.x, st);
    cp_async_commit();
  }
  cp_async_wait<0>();  // only empty groups remain; nothing is left in flight at exit
}

// Signed-integer order keys of binary32 values: the integer order is the float order
// with -0 below +0 (IEEE 754-2019 minimum/maximum); the map is its own inverse.
__device__ __forceinline__ int32_t f32_key(float f) {
  const int32_t b = __float_as_int(f);
  return b ^ ((b >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float f32_unkey(int32_t k) { return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF)); }

// VALUE kind: one lane per kBlk consecutive 16-channel blocks of a row (C = 16 kBlk
// channels; kBlk = 2 when D % 32 == 0 and G >= 32, so a lane's channels lie in one
// group), kRowsPerWarp = 32 / L rows per warp; a group spans W = min(G/C, L) aligned
// lanes, reduced with a xor butterfly of uniform width.  Each lane holds two rows'
// words (the next row's loads are issued before this row's arithmetic), alternating
// between two register sets.  Rows past the end and lanes past the last block load a
// valid row / block (the last one) and store nothing; a repeated block lies in its own
// group or in one that stores nothing.
template <int L, int kBlk, bool kResidual>
__global__ void __launch_bounds__(kThreads, kBlk == 2 ? 3 : 4) int4_value_kernel(const Int4EncodeParams p) {
  constexpr int kRowsPerWarp = 32 / L;
  constexpr int C = 16 * kBlk;     // channels per lane
  constexpr int NW = 8 * kBlk;     // 32-bit words per lane
  const int lane = threadIdx.x & 31;
  const int sub = lane / L;
  const int nb = p.D / C;
  const bool has = lane % L < nb;
  const int b = has ? lane % L : nb - 1;
  const int W = min(p.G / C, L);
  const int ngv = (p.D + p.G - 1) / p.G;
  const bool lead = has && (C * b) % p.G == 0;  // writes its group's metadata
  const int gidx = (C * b) / p.G;
  const uint32_t total = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H);
  const uint32_t stride = gridDim.x * (kThreads / 32) * kRowsPerWarp;
  if (total == 0u) return;

  // the C values of this lane's blocks of row min(rw, total - 1); r = its compact row
  auto load = [&](uint32_t rw, uint32_t (&w)[NW], int32_t& r) {
    uint32_t ru, hu;
    p.div_h.divmod(min(rw, total - 1u), ru, hu);
    r = static_cast<int32_t>(ru);
#pragma unroll
    for (int k = 0; k < 2 * kBlk; ++k) {
      uint32_t a[4];
      load_chunk8<kResidual>(p, r, static_cast<int32_t>(hu), C * b + 8 * k, a);
#pragma unroll
      for (int i = 0; i < 4; ++i) w[4 * k + i] = a[i];
    }
  };

  auto code = [&](uint32_t rw, const uint32_t (&w)[NW], int32_t r) {
    const bool store = rw < total && has;
    if constexpr (kResidual) {
      if (store && b == 0 && static_cast<uint32_t>(r) * static_cast<uint32_t>(p.H) == rw) check_pos<kResidual>(p, r);
    }
    // the lane's minimum / maximum (bf16x2 min/max, sign-OR for a zero minimum), then
    // the group's over W lanes in order keys
    uint32_t m = w[0], M = w[0], s = w[0];
#pragma unroll
    for (int i = 1; i < NW; ++i) {
      m = hmin2(m, w[i]);
      M = hmax2(M, w[i]);
      s |= w[i];
    }
    m = hmin2(m, __byte_perm(m, 0u, 0x1032));  // both halves: the lane's extremes
    M = hmax2(M, __byte_perm(M, 0u, 0x1032));
    int32_t kmn = f32_key(group_min(m, s & 0x80008000u)), kmx = f32_key(bf16lo(M));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      if (o < W) {  // W is uniform: every lane runs the same shuffles
        kmn = min(kmn, __shfl_xor_sync(0xFFFFFFFFu, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(0xFFFFFFFFu, kmx, o));
      }
    }
    const float mn = f32_unkey(kmn);
    const float sc = int4_scale(__fsub_rn(f32_unkey(kmx), mn));
    const uint64_t nmn2[4] = {dup_f32x2(-mn), dup_f32x2(-mn), dup_f32x2(-mn), dup_f32x2(-mn)};
    const uint64_t nsc2[4] = {dup_f32x2(-sc), dup_f32x2(-sc), dup_f32x2(-sc), dup_f32x2(-sc)};
    const float yv = int4_recip(sc);
    const uint64_t y2[4] = {dup_f32x2(yv), dup_f32x2(yv), dup_f32x2(yv), dup_f32x2(yv)};
    const bool fast = int4_fast_scale(sc);
    uint32_t cw[2 * kBlk];
#pragma unroll
    for (int k = 0; k < 2 * kBlk; ++k) {
      const uint32_t wk[4] = {w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]};
      cw[k] = fast ? int4_codes8(wk, nmn2, nsc2, y2) : int4_codes8_div(wk, nmn2, nsc2);
    }
    if (store) {
      uint8_t* const dst = p.dst.codes + static_cast<int64_t>(rw) * (p.D / 2) + (C / 2) * b;
      if constexpr (kBlk == 2) {
        store16B(dst, cw);
      } else {
        store8B(dst, cw[0], cw[1]);
      }
      if (lead) {
        const int64_t mi = static_cast<int64_t>(rw) * ngv + gidx;
        STX(p.dst.mn + mi, f32_to_f16_bits(mn));
        STX(p.dst.sc + mi, f32_to_f16_bits(sc));
      }
    }
  };

  uint32_t row = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
  uint32_t wa[NW], wb[NW];
  int32_t ra, rb;
  load(row, wa, ra);
  while (row - sub < total) {  // row - sub is uniform across the warp
    load(row + stride, wb, rb);
    code(row, wa, ra);
    row += stride;
    if (row - sub >= total) break;
    load(row + stride, wa, ra);
    code(row, wb, rb);
    row += stride;
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

template <int L, int kBlk, bool kRes>
cudaError_t value_launch(const Int4EncodeParams& p, cudaStream_t s) {
  auto k = int4_value_kernel<L, kBlk, kRes>;
  int grid = grid_cap(k, static_cast<int64_t>(p.rows) * p.H, (kThreads / 32) * (32 / L));
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("int4_value_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

template <int kBlk, bool kRes>
cudaError_t value_dispatch_blk(const Int4EncodeParams& p, cudaStream_t s) {
  int nb = p.D / (16 * kBlk), L = 1;
  while (L < nb) L <<= 1;
  switch (L) {
    case 1: return value_launch<1, kBlk, kRes>(p, s);
    case 2: return value_launch<2, kBlk, kRes>(p, s);
    case 4: return value_launch<4, kBlk, kRes>(p, s);
    case 8: return value_launch<8, kBlk, kRes>(p, s);
    case 16: return value_launch<16, kBlk, kRes>(p, s);
    case 32: return value_launch<32, kBlk, kRes>(p, s);
  }
  return cudaErrorInvalidValue;
}

// Two blocks per lane when a lane's 32 channels stay inside one group.
template <bool kRes>
cudaError_t value_dispatch(const Int4EncodeParams& p, cudaStream_t s) {
  if (p.D % 32 == 0 && p.G >= 32) return value_dispatch_blk<2, kRes>(p, s);
  return value_dispatch_blk<1, kRes>(p, s);
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

// Shared memory of the tile kernel: kStages x planes tiles of G x D bf16, the
// [3][RP][D/8] partial chunks and the [3][D/2] float2 group parameters.
size_t key_tile_smem(int G, int D, int stages, int planes) {
  const size_t nchunk = static_cast<size_t>(D / 8);
  return static_cast<size_t>(stages) * planes * G * D * 2 + 3 * (kThreads / nchunk) * nchunk * 16 +
         3 * static_cast<size_t>(D / 2) * 8;
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
  if (key_tile_smem(p.G, p.D, 2, planes) <= kTileSmemCap) return key_tile_launch<kRes, 2>(p, s);
  if (key_tile_smem(p.G, p.D, 1, planes) <= kTileSmemCap) return key_tile_launch<kRes, 1>(p, s);
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
