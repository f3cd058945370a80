// int4_kernels.cu -- INT4 affine codec encode kernels (plain pack and residual).
//
// Format ("vllm-rlt PR #166: INT4 KV packing/unpacking and cross-loop residual
// reconstruction", Purpose, and the review by 0z5a): groups of G values share an
// FP16 minimum and an FP16 scale; the codes come from the FP32 minimum and scale, and
// only then is the metadata rounded to FP16; K groups span G token rows at a fixed
// (head, channel), V groups G channels at a fixed (token, head); the last group may
// be short.  Per group, in order
// (binary32, nearest even):
//   mn = min x;  mx = max x;  sc = (mx - mn) / 15
//   code = 0 if sc == 0, else clamp(rint((x - mn) / sc), 0, 15)   (rint: ties even)
//   stored: fp16(mn), fp16(sc); two codes per byte, low nibble = even channel.
// The minimum and maximum order -0 below +0 (IEEE 754-2019 minimum/maximum).
// Residual encode feeds the same codec with r = bf16(cur - prev) of the kept rows
// (same page, Purpose: a residual is taken against the reconstruction of the
// previous loop, in bf16; K groups follow the order of the packed rows).
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
      w[i] = bf16x2_sub(w[i], q[i]);
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

// KEY kind, in registers: a column task is (group of G rows, head, 8-channel chunk).
// S = G / RPT lanes share a task, lane rs holding rows rs, rs + S, ... (RPT of them) of
// the chunk, so every row is read once.  The lanes' minima, maxima (bf16x2 min/max)
// and sign ORs meet in a xor butterfly; a zero minimum takes its sign from the group's
// OR (a zero minimum means no element is negative, so a set sign bit is a -0).  Every
// lane then forms the 8 channels' parameters and codes its rows.  Rows past a partial
// group repeat its last row and lanes past the last task repeat that task: neither
// changes a group's extrema, and neither stores.
//
// The rows arrive through a per-warp shared-memory slot of RPT x 32 16-byte cells per
// plane (lane l's row k at cell k * 32 + l): each lane copies its own cells with
// cp.async and reads back only those, so the lane's own wait_group orders them and no
// barrier is needed.  The next task's copies are issued once this task's cells have
// been read into registers (the extrema depend on every read, and a warp issues in
// order), so they travel while this task is coded.  Residual mode copies cur and prev
// and forms bf16(cur - prev) on reading; a bad position fills zeros.
template <bool kResidual>
__host__ __device__ constexpr int key_threads() { return kResidual ? 128 : 256; }
template <bool kResidual, int RPT>
__host__ __device__ constexpr size_t key_smem() { return static_cast<size_t>(key_threads<kResidual>() / 32) * (kResidual ? 2 : 1) * RPT * 32 * 16; }

template <bool kResidual, int S, int RPT>
__global__ void __launch_bounds__(key_threads<kResidual>(), kResidual ? 4 : 2) int4_key_kernel(const Int4EncodeParams p) {
  constexpr int kWarps = key_threads<kResidual>() / 32;
  constexpr int CW = 32 / S;  // column tasks per warp
  extern __shared__ __align__(16) unsigned char smem[];
  uint4* const slot = reinterpret_cast<uint4*>(smem) + (threadIdx.x / 32) * ((kResidual ? 2 : 1) * RPT * 32);
  const int lane = threadIdx.x & 31;
  const int rs = lane / CW;
  const int cl = lane % CW;
  const int32_t nchunk = p.D / 8;
  const int32_t ngroups = (p.rows + p.G - 1) / p.G;
  const int64_t ntask = static_cast<int64_t>(ngroups) * p.H * nchunk;
  const int64_t nwtask = (ntask + CW - 1) / CW;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

  struct Task {
    int32_t chunk, h, g, r0, rlast;
    bool valid;
  };
  // task -> (group, head, chunk): multiply-shift divisions while the task count is
  // below 2^31 (always, short of tensors near the memory size), else 64-bit ones
  const bool small = ntask < (int64_t{1} << 31);
  const FastDiv div_c(static_cast<uint32_t>(nchunk));  // built once per thread
  auto task_of = [&](int64_t wt) {
    Task t;
    const int64_t task = wt * CW + cl;
    t.valid = task < ntask;
    const int64_t tk = t.valid ? task : ntask - 1;
    if (small) {
      uint32_t gh, c, g, h;
      div_c.divmod(static_cast<uint32_t>(tk), gh, c);
      p.div_h.divmod(gh, g, h);
      t.chunk = static_cast<int32_t>(c);
      t.h = static_cast<int32_t>(h);
      t.g = static_cast<int32_t>(g);
    } else {
      t.chunk = static_cast<int32_t>(tk % nchunk);
      t.h = static_cast<int32_t>((tk / nchunk) % p.H);
      t.g = static_cast<int32_t>(tk / (static_cast<int64_t>(nchunk) * p.H));
    }
    t.r0 = t.g * p.G;
    t.rlast = min(p.rows, t.r0 + p.G) - 1;
    return t;
  };
  // copies of this lane's rows of warp task wt into the slot (nothing past the end)
  auto issue = [&](int64_t wt) {
    if (wt >= nwtask) return;  // uniform across the warp
    const Task t = task_of(wt);
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      uint4* const cell = slot + k * 32 + lane;
      int64_t src = min(t.r0 + rs + k * S, t.rlast);
      if constexpr (kResidual) {
        if (p.pos != nullptr) src = LDX(p.pos + src);
        if (src < 0 || src >= p.src_rows) {
          *cell = make_uint4(0u, 0u, 0u, 0u);
          cell[RPT * 32] = make_uint4(0u, 0u, 0u, 0u);
          continue;
        }
        cp_async16(cell + RPT * 32,
                   p.prev + src * p.prev_row_pitch + static_cast<int64_t>(t.h) * p.prev_head_pitch + t.chunk * 8);
      }
      cp_async16(cell, p.x + src * p.row_pitch + static_cast<int64_t>(t.h) * p.head_pitch + t.chunk * 8);
    }
  };

  int64_t wt = blockIdx.x * static_cast<int64_t>(kWarps) + threadIdx.x / 32;
  issue(wt);
  cp_async_commit();
  for (; wt < nwtask; wt += nwarps) {
    cp_async_wait<0>();
    const Task t = task_of(wt);
    uint32_t v[RPT][4];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      uint4 a = slot[k * 32 + lane];
      if constexpr (kResidual) {
        const uint4 q = slot[(RPT + k) * 32 + lane];
        a.x = bf16x2_sub(a.x, q.x);
        a.y = bf16x2_sub(a.y, q.y);
        a.z = bf16x2_sub(a.z, q.z);
        a.w = bf16x2_sub(a.w, q.w);
      }
      v[k][0] = a.x;
      v[k][1] = a.y;
      v[k][2] = a.z;
      v[k][3] = a.w;
    }
    // the lane's minima, maxima and sign ORs over its RPT rows, as pairwise trees
    uint32_t m[4], M[4], sg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t tm[RPT / 2], tM[RPT / 2], ts[RPT / 2];
#pragma unroll
      for (int k = 0; k < RPT / 2; ++k) {
        tm[k] = hmin2(v[2 * k][i], v[2 * k + 1][i]);
        tM[k] = hmax2(v[2 * k][i], v[2 * k + 1][i]);
        ts[k] = v[2 * k][i] | v[2 * k + 1][i];
      }
#pragma unroll
      for (int w = RPT / 4; w >= 1; w /= 2) {
#pragma unroll
        for (int k = 0; k < w; ++k) {
          tm[k] = hmin2(tm[2 * k], tm[2 * k + 1]);
          tM[k] = hmax2(tM[2 * k], tM[2 * k + 1]);
          ts[k] = ts[2 * k] | ts[2 * k + 1];
        }
      }
      m[i] = tm[0];
      M[i] = tM[0];
      sg[i] = ts[0];
    }
    issue(wt + nwarps);  // every cell of this task has been read (the extrema use them all)
    cp_async_commit();
#pragma unroll
    for (int o = CW; o < 32; o <<= 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m[i] = hmin2(m[i], __shfl_xor_sync(0xFFFFFFFFu, m[i], o));
        M[i] = hmax2(M[i], __shfl_xor_sync(0xFFFFFFFFu, M[i], o));
        sg[i] |= __shfl_xor_sync(0xFFFFFFFFu, sg[i], o);
      }
    }
    // parameters: lane rs forms those of words rs, rs + S, ... (every lane of a task
    // holds the same extrema), then each word's come from the lane that formed them
    constexpr int WPL = S >= 4 ? 1 : 4 / S;  // words whose parameters this lane forms
    uint64_t pn[WPL], ps[WPL], py[WPL];
    uint32_t pm16[WPL], ps16[WPL];
    bool fast = true;
#pragma unroll
    for (int j = 0; j < WPL; ++j) {
      const int i = S >= 4 ? rs % 4 : rs + j * S;
      uint32_t mi = m[0], Mi = M[0], si = sg[0];
#pragma unroll
      for (int q = 1; q < 4; ++q) {  // select word i without dynamic register indexing
        if (i == q) {
          mi = m[q];
          Mi = M[q];
          si = sg[q];
        }
      }
      const float mnl = group_min(mi, si & 0x8000u), mnh = group_min(mi >> 16, si & 0x80000000u);
      const float scl = int4_scale(__fsub_rn(bf16lo(Mi), mnl)), sch = int4_scale(__fsub_rn(bf16hi(Mi), mnh));
      pn[j] = pack_f32x2(__float_as_uint(-mnl), __float_as_uint(-mnh));
      ps[j] = pack_f32x2(__float_as_uint(-scl), __float_as_uint(-sch));
      py[j] = pack_f32x2(__float_as_uint(int4_recip(scl)), __float_as_uint(int4_recip(sch)));
      pm16[j] = static_cast<uint32_t>(f32_to_f16_bits(mnl)) | (static_cast<uint32_t>(f32_to_f16_bits(mnh)) << 16);
      ps16[j] = static_cast<uint32_t>(f32_to_f16_bits(scl)) | (static_cast<uint32_t>(f32_to_f16_bits(sch)) << 16);
      fast = fast && int4_fast_scale(scl) && int4_fast_scale(sch);
    }
    int fast_all = fast ? 1 : 0;  // AND over the lanes that formed parameters (every lane shuffles)
#pragma unroll
    for (int o = CW; o < CW * (S < 4 ? S : 4); o <<= 1) fast_all &= __shfl_xor_sync(0xFFFFFFFFu, fast_all, o);
    fast = fast_all != 0;
    uint64_t nmn[4], nsc[4], y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int src = (S >= 4 ? i : i % S) * CW + cl;
      const int j = S >= 4 ? 0 : i / S;
      nmn[i] = __shfl_sync(0xFFFFFFFFu, pn[j], src);
      nsc[i] = __shfl_sync(0xFFFFFFFFu, ps[j], src);
      y[i] = __shfl_sync(0xFFFFFFFFu, py[j], src);
    }
    const int32_t col = t.chunk * 8;
    uint8_t* const cbase = p.dst.codes + static_cast<int64_t>(t.h) * (p.D / 2) + col / 2;
    const int64_t cstride = static_cast<int64_t>(p.H) * (p.D / 2);
    if (fast && t.valid && t.r0 + rs + (RPT - 1) * S <= t.rlast) {  // every row, ordinary scales: unrolled
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        const int32_t r = t.r0 + rs + k * S;
        if (t.chunk == 0 && t.h == 0) check_pos<kResidual>(p, r);
        STX(reinterpret_cast<uint32_t*>(cbase + r * cstride), int4_codes8(v[k], nmn, nsc, y));
      }
    } else if (t.valid) {  // a partial group or a scale below 2^-64: compact, rows read again
#pragma unroll 1
      for (int32_t r = t.r0 + rs; r <= t.rlast; r += S) {
        uint32_t wk[4];
        load_chunk8<kResidual>(p, r, t.h, col, wk);
        if (t.chunk == 0 && t.h == 0) check_pos<kResidual>(p, r);
        STX(reinterpret_cast<uint32_t*>(cbase + r * cstride),
            fast ? int4_codes8(wk, nmn, nsc, y) : int4_codes8_div(wk, nmn, nsc));
      }
    }
    if (t.valid && rs < 4) {  // the FP16 metadata of the words this lane formed
      const int64_t mi = (static_cast<int64_t>(t.g) * p.H + t.h) * p.D + col;
#pragma unroll
      for (int j = 0; j < WPL; ++j) {
        const int i = S >= 4 ? rs : rs + j * S;
        STX(reinterpret_cast<uint32_t*>(p.dst.mn + mi + 2 * i), pm16[j]);
        STX(reinterpret_cast<uint32_t*>(p.dst.sc + mi + 2 * i), ps16[j]);
      }
    }
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
    uint32_t tm[NW / 2], tM[NW / 2], ts[NW / 2];  // pairwise trees over the lane's words
#pragma unroll
    for (int k = 0; k < NW / 2; ++k) {
      tm[k] = hmin2(w[2 * k], w[2 * k + 1]);
      tM[k] = hmax2(w[2 * k], w[2 * k + 1]);
      ts[k] = w[2 * k] | w[2 * k + 1];
    }
#pragma unroll
    for (int n = NW / 4; n >= 1; n /= 2) {
#pragma unroll
      for (int k = 0; k < n; ++k) {
        tm[k] = hmin2(tm[2 * k], tm[2 * k + 1]);
        tM[k] = hmax2(tM[2 * k], tM[2 * k + 1]);
        ts[k] = ts[2 * k] | ts[2 * k + 1];
      }
    }
    uint32_t m = tm[0], M = tM[0], s = ts[0];
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
    uint8_t* const dst = p.dst.codes + static_cast<int64_t>(rw) * (p.D / 2) + (C / 2) * b;
    if (int4_fast_scale(sc)) {
      uint32_t cw[2 * kBlk];
#pragma unroll
      for (int k = 0; k < 2 * kBlk; ++k) {
        const uint32_t wk[4] = {w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]};
        cw[k] = int4_codes8(wk, nmn2, nsc2, y2);
      }
      if (store) {
        if constexpr (kBlk == 2) {
          store16B(dst, cw);
        } else {
          store8B(dst, cw[0], cw[1]);
        }
      }
    } else if (store) {  // a scale below 2^-64: divide, compact, the chunks read again
      const int32_t h = static_cast<int32_t>(rw - static_cast<uint32_t>(r) * static_cast<uint32_t>(p.H));
#pragma unroll 1
      for (int k = 0; k < 2 * kBlk; ++k) {
        uint32_t wk[4];
        load_chunk8<kResidual>(p, r, h, C * b + 8 * k, wk);
        STX(reinterpret_cast<uint32_t*>(dst + 4 * k), int4_codes8_div(wk, nmn2, nsc2));
      }
    }
    if (store) {
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

// Resident blocks per SM of a kernel instance, with its dynamic shared memory opted in
// first; computed once per device (0: the opt-in failed).
template <auto Kernel>
int occupancy(int threads, size_t smem) {
  constexpr int kDevices = 64;
  static int cache[kDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kDevices) dev = 0;
  if (cache[dev] == 0) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
      return 0;
    int o = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, Kernel, threads, smem);
    cache[dev] = o < 1 ? 1 : o;
  }
  return cache[dev];
}

// Blocks for `work_items` items at `items_per_cta` each, at most one wave.
int grid_for(int occ, int64_t work_items, int items_per_cta) {
  int64_t need = (work_items + items_per_cta - 1) / items_per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms()) * occ;
  if (need < 1) need = 1;
  return static_cast<int>(need < cap ? need : cap);
}

template <int L, int kBlk, bool kRes>
cudaError_t value_launch(const Int4EncodeParams& p, cudaStream_t s) {
  auto k = int4_value_kernel<L, kBlk, kRes>;
  const int grid = grid_for(occupancy<int4_value_kernel<L, kBlk, kRes>>(kThreads, 0),
                            static_cast<int64_t>(p.rows) * p.H, (kThreads / 32) * (32 / L));
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

template <bool kRes, int S, int RPT>
cudaError_t key_launch(const Int4EncodeParams& p, int64_t ntask, cudaStream_t s) {
  auto k = int4_key_kernel<kRes, S, RPT>;
  constexpr int threads = key_threads<kRes>();
  constexpr size_t smem = key_smem<kRes, RPT>();
  const int occ = occupancy<int4_key_kernel<kRes, S, RPT>>(threads, smem);
  if (occ == 0) return cudaErrorInvalidValue;
  const int grid = grid_for(occ, (ntask + 32 / S - 1) / (32 / S), threads / 32);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("int4_key_kernel", s, k<<<grid, threads, smem, s>>>(p); e = cudaGetLastError());
  return e;
}

template <bool kRes>
cudaError_t key_dispatch(const Int4EncodeParams& p, cudaStream_t s) {
  const int64_t ntask = static_cast<int64_t>((p.rows + p.G - 1) / p.G) * p.H * (p.D / 8);
  if constexpr (kRes) {
    switch (p.G) {  // S = G / RPT lanes per column task, RPT rows each (8; 16 for G512)
      case 16: return key_launch<kRes, 2, 8>(p, ntask, s);
      case 32: return key_launch<kRes, 4, 8>(p, ntask, s);
      case 64: return key_launch<kRes, 8, 8>(p, ntask, s);
      case 128: return key_launch<kRes, 16, 8>(p, ntask, s);
      case 256: return key_launch<kRes, 32, 8>(p, ntask, s);
      case 512: return key_launch<kRes, 32, 16>(p, ntask, s);
    }
  } else {
    switch (p.G) {  // S = G / 16 lanes per column task, 16 rows each
      case 16: return key_launch<kRes, 1, 16>(p, ntask, s);
      case 32: return key_launch<kRes, 2, 16>(p, ntask, s);
      case 64: return key_launch<kRes, 4, 16>(p, ntask, s);
      case 128: return key_launch<kRes, 8, 16>(p, ntask, s);
      case 256: return key_launch<kRes, 16, 16>(p, ntask, s);
      case 512: return key_launch<kRes, 32, 16>(p, ntask, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_int4_encode(const Int4EncodeParams& p, cudaStream_t s) {
  if (p.kind == 0) return p.residual ? key_dispatch<true>(p, s) : key_dispatch<false>(p, s);
  return p.residual ? value_dispatch<true>(p, s) : value_dispatch<false>(p, s);
}

}  // namespace kvq
