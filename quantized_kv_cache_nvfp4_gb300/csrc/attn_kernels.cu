// attn_kernels.cu -- paged decode attention that reads the quantised pool directly.
//
// The step downstream of the paged restore: instead of restoring K and V to bf16,
// decode attention dequantises them in registers ("feat(kvcache): add nvfp4 kv
// quantization (FreeToken PR #408)", Summary -- the restore paths -- and fp8 store
// notes, where the row scale multiplies the score and the output; "vllm-rlt PR #166",
// review by 0z5a: dequantise to 16 bits in registers and keep the 16-bit MMA).
//
// One query token per sequence; query head qh reads KV head qh / group:
//   o[s][qh] = softmax_t(scale * q . k_t) . v_t   over tokens t < seq_lens[s].
//
// Mapping (mma.sync m16n8k16, f16 operands, f32 accumulators), token-major.  A CTA
// takes one (split of a sequence's tokens, KV head, sequence); its 4 warps take
// 16-token tiles in turn, each through its own cp.async ring of pool tiles in shared
// memory.
//  * M = the tile's 16 tokens, N = the group's query heads in n-tiles of 8 (one for
//    groups up to 8, two up to 16): a warp computes S^T = K Q^T, 16 tokens x 8 heads
//    per n-tile, with K as the A operand, so no MMA row is padding.
//  * S^T contracts over the head dimension in a permuted order: k-step kb of lane c
//    (c = lane % 4) covers dims c*D/4 + 4kb .. + 3, so a lane's K operand for one token
//    is one contiguous run of code bytes; Q^T is permuted the same way and stays in
//    registers when its fragments fit in 16 of them (D = 64, or D = 128 with one
//    n-tile), else it is read from shared memory per k-step.
//  * The probabilities leave the S^T accumulators in the C layout (a lane holds two
//    heads of tokens g and g + 8); an 8x8 transpose in registers (movmatrix) turns
//    them into the B operand of O^T = V^T P^T (two tokens of one head).
//  * O^T: m-tile mt, rows g and g + 8 = dims g*D/8 + 2mt and + 1, so a lane's V operand
//    for one token is again one contiguous run; the nibbles (or bytes) of the two
//    tokens a register pairs are interleaved by a mask-and-shift (or byte-permute)
//    transpose.
//  * K and V decode exactly to f16: e2m1 x e4m3 has at most 2 x 4 significant bits,
//    and e4m3 fits f16.  K's FP32 row scale multiplies the score; V's multiplies P
//    relative to a reference R of the tile row scales.  R and the softmax reference m
//    move only when a tile exceeds them by more than 2^6 and 2^8 (O is rescaled then),
//    so P' = exp2(s - m) * rs / R stays below 2^14 and f16 holds it.
//  * Q enters f16 exactly: each query row is scaled by a power of two that puts its
//    largest element in [2^14, 2^15), undone in the score multiplier.
//  * The warps of a CTA merge through shared memory; several splits of a sequence
//    merge through the caller's workspace in a second small kernel.
#include <atomic>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Both E4M3 bytes of `two` (low byte -> low half) to f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  const uint16_t in = static_cast<uint16_t>(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  return r;
}

// The four E2M1 pairs of a word, byte i -> f16x2 i (low nibble in the low half),
// exactly; the bytes go to the conversions as .b8 registers (no shifts or masks).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// The two E4M3 pairs of a word, bytes 0-1 -> f16x2 0 and bytes 2-3 -> f16x2 1, exactly.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t (&h)[2]) {
  asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, u;\n\t}"
      : "=r"(h[0]), "=r"(h[1])
      : "r"(w));
}

__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// The same with results below 2^-126 flushed to zero: used for probabilities, whose
// row sum is at least 1, so a flushed term is below the sum's own rounding.
__device__ __forceinline__ float ex2_ftz(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Asynchronous 4- / 8-byte copies into shared memory (cp.async.ca; 16-byte copies use
// cp_async16).  The checked build stores zeros instead of copying from outside a
// registered range.
template <int N>
__device__ __forceinline__ void cp_async_small(void* smem_dst, const void* gsrc) {
  static_assert(N == 4 || N == 8, "4 or 8 bytes");
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  if (!KVQ_OK(gsrc, N, N)) {
    if constexpr (N == 4) {
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(d), "r"(0u) : "memory");
    } else {
      asm volatile("st.shared.v2.b32 [%0], {%1, %1};" ::"r"(d), "r"(0u) : "memory");
    }
    return;
  }
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(d), "l"(gsrc), "n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_n(void* smem_dst, const void* gsrc) {
  if constexpr (N == 16) {
    cp_async16(smem_dst, gsrc);
  } else {
    cp_async_small<N>(smem_dst, gsrc);
  }
}

__device__ __forceinline__ int64_t shfl64(int64_t v, int src) {
  const int lo = __shfl_sync(0xFFFFFFFFu, static_cast<int>(v & 0xFFFFFFFF), src);
  const int hi = __shfl_sync(0xFFFFFFFFu, static_cast<int>(v >> 32), src);
  return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

// Shared-memory layout of one 16-token tile of one KV head (both K and V).  Row
// strides are chosen so that each access phase of a warp covers 32 distinct banks:
// a K read is one lane's contiguous chunk (D/8 or D/4 bytes at lane c's offset) of
// token 8j + g; a V read is D/16 or D/8 bytes at lane g's offset of token 2c (+1,
// +8, +9), which needs a row stride of 4 mod 16 words (the code bytes + 16).
template <int D, int kFK, int kFV>
struct AttnTile {
  static constexpr int kCK = kFK == 3 ? D : D / 2;  // code bytes per row
  static constexpr int kCV = kFV == 3 ? D : D / 2;
  static constexpr int kSK = kFK == 3 ? (D == 128 ? 144 : D) : (D == 256 ? 144 : D / 2);  // smem row strides
  static constexpr int kSV = kCV + 16;
  static constexpr int kBK = kFK == 3 ? 0 : D / 16;  // block-scale bytes per row
  static constexpr int kBV = kFV == 3 ? 0 : D / 16;
  static constexpr int kOffKC = 0;
  static constexpr int kOffVC = kOffKC + 16 * kSK;
  static constexpr int kOffKB = kOffVC + 16 * kSV;
  static constexpr int kOffVB = kOffKB + 16 * kBK;
  static constexpr int kOffKR = kOffVB + 16 * kBV;
  static constexpr int kOffVR = kOffKR + 64;
  static constexpr int kBytes = kOffVR + 64;
  static constexpr int kStages = kBytes > 4096 ? 3 : 4;
  static constexpr int kRing = kAttnWarps * kStages * kBytes;
  // per warp: up to 16 query heads x (O, m, l); Q^T fragments [n-tile][k-step][lane]
  // (8 B each, up to two n-tiles) + up to 16 head factors
  static constexpr int kMerge = kAttnWarps * 16 * (D + 2) * 4;
  static constexpr int kQ = (D / 16) * 32 * 16 + 64;
  static constexpr int kSmem = kQ + (kRing > kMerge ? kRing : kMerge);
};

// NW words from shared memory at p (aligned to the access), in 16-, 8- or 4-byte loads.
template <int NW>
__device__ __forceinline__ void lds_words(const unsigned char* p, uint32_t (&w)[NW]) {
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  } else if constexpr (NW == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

// Transpose of an 8x8 f16 matrix held as one m16n8 fragment quarter: lane (g, c) gives
// row g, columns 2c and 2c + 1, and receives row g, columns 2c and 2c + 1 of the
// transpose.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Shared-memory view of one 16-token tile of one KV head: the code, block-scale and row
// scale rows of token i start at kc / vc / kb / vb / kr / vr + i * stride (bytes).
struct TileView {
  const unsigned char *kc, *vc, *kb, *vb, *kr, *vr;
  int sk, sv, sbk, sbv, sr;
};

// A warp's running softmax state over its tiles: per head (8nh + 2c + e) the reference
// m (and m + 8), the partial sum l of this lane's tokens, the V row-scale reference R
// (R64 = 64 R, rR = 1 / R), and the O^T accumulators o[mt][nh] (dims g*D/8 + 2mt,
// e = 0, 1, and + 1, e = 2, 3, of heads 8nh + 2c and + 1), relative to R.
template <int D, int kNH>
struct AttnState {
  float m[kNH][2], m8[kNH][2], l[kNH][2], R, R64, rR;
  float o[D / 16][kNH][4];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) {
      m[nh][0] = m[nh][1] = m8[nh][0] = m8[nh][1] = kNegInf;
      l[nh][0] = l[nh][1] = 0.0f;
    }
    R = R64 = rR = 0.0f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh) o[mt][nh][0] = o[mt][nh][1] = o[mt][nh][2] = o[mt][nh][3] = 0.0f;
  }
};

// One 16-token tile of one KV head into the warp's state: S^T = K Q^T, the softmax
// update, O^T += V^T P'^T.  nvalid = tokens of the tile inside the sequence (16 but on
// a split's last tile).  qb(nh, kb) gives the Q^T fragment, qmul the per-head query
// factors (scale, log2 e, Q's power of two).
template <int D, int kFK, int kFV, int kNH, typename QB>
__device__ __forceinline__ void attn_tile(const TileView& tv, const QB& qb, const float (&qmul)[kNH][2], int lane,
                                          int nvalid, AttnState<D, kNH>& st) {
  constexpr int kKS = D / 16;
  constexpr int kMT = D / 16;
  const int g = lane >> 2;
  const int c = lane & 3;
  // S^T = K Q^T: rows g and g + 8 are tokens g and 8 + g (this lane's K rows), each
  // K fragment serves every head n-tile
  float sc[kNH][4];
#pragma unroll
  for (int nh = 0; nh < kNH; ++nh) sc[nh][0] = sc[nh][1] = sc[nh][2] = sc[nh][3] = 0.0f;
  if constexpr (kFK == 3) {
    uint32_t kw[2][D / 16];  // this lane's D/4 code bytes of tokens g and 8 + g
    lds_words<D / 16>(tv.kc + g * tv.sk + c * (D / 4), kw[0]);
    lds_words<D / 16>(tv.kc + (8 + g) * tv.sk + c * (D / 4), kw[1]);
#pragma unroll
    for (int kb = 0; kb < kKS; ++kb) {
      uint32_t k0[2], k1[2];
      e4m3x4_to_f16x2(kw[0][kb], k0);  // dims 4kb, 4kb+1 | 4kb+2, 4kb+3
      e4m3x4_to_f16x2(kw[1][kb], k1);
      const uint32_t a[4] = {k0[0], k1[0], k0[1], k1[1]};
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh) {
        const uint2 b = qb(nh, kb);
        mma_f16_16816(sc[nh], a, b.x, b.y);
      }
    }
  } else {
    uint32_t kw[2][D / 32];  // this lane's D/8 code bytes of tokens g and 8 + g
    lds_words<D / 32>(tv.kc + g * tv.sk + c * (D / 8), kw[0]);
    lds_words<D / 32>(tv.kc + (8 + g) * tv.sk + c * (D / 8), kw[1]);
    constexpr int kNB = D / 64 > 0 ? D / 64 : 1;  // blocks of this lane's dims
    uint32_t bsb[2][kNB];                         // their scales, f16 in both halves
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint8_t* kbs = tv.kb + (8 * j + g) * tv.sbk + c * (D / 64);
      if constexpr (kNB == 1) {
        const uint32_t bsh = e4m3_to_f16x2(kbs[0]) & 0xFFFFu;
        bsb[j][0] = bsh | (bsh << 16);
      } else {  // pairs of scale bytes, one conversion each, halves spread by a permute
#pragma unroll
        for (int i = 0; i < kNB; i += 2) {
          const uint32_t two = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(kbs + i));
          bsb[j][i] = __byte_perm(two, 0u, 0x1010);
          bsb[j][i + 1] = __byte_perm(two, 0u, 0x3232);
        }
      }
    }
#pragma unroll
    for (int wi = 0; wi < D / 32; ++wi) {  // one code word = k-steps 2wi and 2wi + 1
      uint32_t hk[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        e2m1x8_to_f16x2(kw[j][wi], hk[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) hk[j][i] = hmul2(hk[j][i], bsb[j][(2 * wi) / 4]);
      }
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        const uint32_t a[4] = {hk[0][2 * hs], hk[1][2 * hs], hk[0][2 * hs + 1], hk[1][2 * hs + 1]};
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh) {
          const uint2 b = qb(nh, 2 * wi + hs);
          mma_f16_16816(sc[nh], a, b.x, b.y);
        }
      }
    }
  }
  // scores times K's row scale; the query factor (scale, log2 e, Q's power of two,
  // positive) enters with the reference in one FMA below, and the maxima are scaled
  // by it once.  Tokens past the end are masked (only a split's last tile can hold
  // any).
  const float kr0 = *reinterpret_cast<const float*>(tv.kr + g * tv.sr);
  const float kr1 = *reinterpret_cast<const float*>(tv.kr + (g + 8) * tv.sr);
  const float vr0 = *reinterpret_cast<const float*>(tv.vr + g * tv.sr);
  const float vr1 = *reinterpret_cast<const float*>(tv.vr + (g + 8) * tv.sr);
  const bool dead0 = g >= nvalid, dead1 = g + 8 >= nvalid;  // past the sequence (last tile only)
  // this lane's maxima (two tokens per head) first: the references move when any
  // lane's exceed them, and only then are the tile's maxima reduced across lanes
  float mt[kNH][2];
  bool move = false;
#pragma unroll
  for (int nh = 0; nh < kNH; ++nh) {
    sc[nh][0] *= kr0;
    sc[nh][1] *= kr0;
    sc[nh][2] *= kr1;
    sc[nh][3] *= kr1;
  }
  if (nvalid < 16) {  // uniform: the tile ends inside the sequence
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) {
      if (dead0) sc[nh][0] = sc[nh][1] = kNegInf;
      if (dead1) sc[nh][2] = sc[nh][3] = kNegInf;
    }
  }
#pragma unroll
  for (int nh = 0; nh < kNH; ++nh) {
    mt[nh][0] = fmaxf(sc[nh][0], sc[nh][2]) * qmul[nh][0];
    mt[nh][1] = fmaxf(sc[nh][1], sc[nh][3]) * qmul[nh][1];
    move = move || mt[nh][0] > st.m8[nh][0] || mt[nh][1] > st.m8[nh][1];
  }
  float rmax = fmaxf(vr0, vr1);
  move = move || rmax > st.R64;
  // references: the softmax reference m per head and the V row-scale reference st.R
  // move only when a tile exceeds them by more than 2^8 and 2^6, so P' = exp2(s - m)
  // * rs_v / st.R stays below 2^14 (f16 holds it) and O is rescaled on few tiles
  if (__any_sync(0xFFFFFFFFu, move)) {
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
#pragma unroll
      for (int nh = 0; nh < kNH; ++nh) {
        mt[nh][0] = fmaxf(mt[nh][0], __shfl_xor_sync(0xFFFFFFFFu, mt[nh][0], off));
        mt[nh][1] = fmaxf(mt[nh][1], __shfl_xor_sync(0xFFFFFFFFu, mt[nh][1], off));
      }
      rmax = fmaxf(rmax, __shfl_xor_sync(0xFFFFFFFFu, rmax, off));
    }
    const float Rn = fmaxf(fmaxf(st.R, rmax), 0x1p-126f);
    const float rr = st.R / Rn;
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float mn = fmaxf(st.m[nh][e], mt[nh][e]);
        const float a = ex2(st.m[nh][e] - mn);  // 0 while m is -inf
        const float f = a * rr;
#pragma unroll
        for (int q = 0; q < kMT; ++q) {
          st.o[q][nh][e] *= f;
          st.o[q][nh][e + 2] *= f;
        }
        st.l[nh][e] *= a;
        st.m[nh][e] = mn;
        st.m8[nh][e] = mn + 8.0f;
      }
    }
    st.R = Rn;
    st.R64 = Rn * 64.0f;
    st.rR = rcp_approx(Rn);
  }
  // P'^T = exp2(s - m) * rs_v / st.R, transposed in registers into the B operand of
  // O^T += V^T P'^T: pb[nh][0] holds tokens 2c, 2c + 1 of head 8nh + g, pb[nh][1]
  // tokens 2c + 8, 2c + 9
  const float r0 = vr0 * st.rR, r1 = vr1 * st.rR;
  uint32_t pb[kNH][2];
#pragma unroll
  for (int nh = 0; nh < kNH; ++nh) {
    const float p0 = ex2_ftz(__fmaf_rn(sc[nh][0], qmul[nh][0], -st.m[nh][0]));  // token g
    const float p1 = ex2_ftz(__fmaf_rn(sc[nh][1], qmul[nh][1], -st.m[nh][1]));
    const float p2 = ex2_ftz(__fmaf_rn(sc[nh][2], qmul[nh][0], -st.m[nh][0]));  // token g + 8
    const float p3 = ex2_ftz(__fmaf_rn(sc[nh][3], qmul[nh][1], -st.m[nh][1]));
    st.l[nh][0] += p0 + p2;
    st.l[nh][1] += p1 + p3;
    pb[nh][0] = transpose8x8(f32x2_to_f16x2(p0 * r0, p1 * r0));
    pb[nh][1] = transpose8x8(f32x2_to_f16x2(p2 * r1, p3 * r1));
  }
  // O^T += V^T P'^T: m-tile mt, rows g and g + 8 = dims g * D/8 + 2mt and + 1; this
  // lane supplies V for tokens (2c, 2c + 1) and (2c + 8, 2c + 9) at those dims
  {
    const int ta0 = 2 * c, ta1 = 2 * c + 8;
    if constexpr (kFV == 3) {
      uint32_t v0[D / 32], v1[D / 32], v2[D / 32], v3[D / 32];  // D/8 bytes of each token
      lds_words<D / 32>(tv.vc + ta0 * tv.sv + g * (D / 8), v0);
      lds_words<D / 32>(tv.vc + (ta0 + 1) * tv.sv + g * (D / 8), v1);
      lds_words<D / 32>(tv.vc + ta1 * tv.sv + g * (D / 8), v2);
      lds_words<D / 32>(tv.vc + (ta1 + 1) * tv.sv + g * (D / 8), v3);
#pragma unroll
      for (int q = 0; q < kMT; ++q) {  // dims 2q, 2q + 1: bytes of one half word
        const int wd = q / 2, bo2 = 2 * (q % 2);
        const uint32_t sel = bo2 | ((4 + bo2) << 4) | ((bo2 + 1) << 8) | ((5 + bo2) << 12);
        uint32_t h01[2], h23[2];
        e4m3x4_to_f16x2(__byte_perm(v0[wd], v1[wd], sel), h01);
        e4m3x4_to_f16x2(__byte_perm(v2[wd], v3[wd], sel), h23);
        const uint32_t a[4] = {h01[0], h01[1], h23[0], h23[1]};
#pragma unroll
        for (int nh = 0; nh < kNH; ++nh) mma_f16_16816(st.o[q][nh], a, pb[nh][0], pb[nh][1]);
      }
    } else {
      constexpr int kW = D / 64;  // code words per lane per token (D/16 bytes)
      uint32_t v0[kW], v1[kW], v2[kW], v3[kW];
      lds_words<kW>(tv.vc + ta0 * tv.sv + g * (D / 16), v0);
      lds_words<kW>(tv.vc + (ta0 + 1) * tv.sv + g * (D / 16), v1);
      lds_words<kW>(tv.vc + ta1 * tv.sv + g * (D / 16), v2);
      lds_words<kW>(tv.vc + (ta1 + 1) * tv.sv + g * (D / 16), v3);
      // block scales of this lane's dims g * D/8 .. + D/8 - 1 for its four tokens: one
      // 16-dim block (D <= 128) or two (D = 256), as f16x2 pairs (tokens ta, ta + 1)
      constexpr int kVB = D / 8 > 16 ? D / 128 : 1;
      const uint8_t* vbs = tv.vb;
      uint32_t bs01[kVB], bs23[kVB];
#pragma unroll
      for (int q = 0; q < kVB; ++q) {
        const int blk = (g * (D / 8)) / 16 + q;
        bs01[q] = e4m3x2_to_f16x2(vbs[ta0 * tv.sbv + blk] | (vbs[(ta0 + 1) * tv.sbv + blk] << 8));
        bs23[q] = e4m3x2_to_f16x2(vbs[ta1 * tv.sbv + blk] | (vbs[(ta1 + 1) * tv.sbv + blk] << 8));
      }
#pragma unroll
      for (int i = 0; i < kW; ++i) {
        // nibble transpose: X byte b = (dim 2(4i+b) of token a | the same dim of token
        // b << 4), Y: the odd dims; then byte b of X / Y is m-tile 4i + b, row g / g + 8
        const uint32_t x01 = (v0[i] & 0x0F0F0F0Fu) | ((v1[i] & 0x0F0F0F0Fu) << 4);
        const uint32_t y01 = ((v0[i] >> 4) & 0x0F0F0F0Fu) | (v1[i] & 0xF0F0F0F0u);
        const uint32_t x23 = (v2[i] & 0x0F0F0F0Fu) | ((v3[i] & 0x0F0F0F0Fu) << 4);
        const uint32_t y23 = ((v2[i] >> 4) & 0x0F0F0F0Fu) | (v3[i] & 0xF0F0F0F0u);
        uint32_t hx01[4], hy01[4], hx23[4], hy23[4];
        e2m1x8_to_f16x2(x01, hx01);
        e2m1x8_to_f16x2(y01, hy01);
        e2m1x8_to_f16x2(x23, hx23);
        e2m1x8_to_f16x2(y23, hy23);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int q = 4 * i + bb;             // m-tile: dims 2q, 2q + 1, one 16-block
          const int vb = kVB == 1 ? 0 : q / 8;  // g * D/8 is a multiple of 16 when D = 256
          const uint32_t a[4] = {hmul2(hx01[bb], bs01[vb]), hmul2(hy01[bb], bs01[vb]),
                                 hmul2(hx23[bb], bs23[vb]), hmul2(hy23[bb], bs23[vb])};
#pragma unroll
          for (int nh = 0; nh < kNH; ++nh) mma_f16_16816(st.o[q][nh], a, pb[nh][0], pb[nh][1]);
        }
      }
    }
  }}

template <int D, int kFK, int kFV, int kNH>
__global__ void __launch_bounds__(kAttnThreads) decode_attn_kernel(const AttnParams p) {
  using T = AttnTile<D, kFK, kFV>;
  constexpr int kKS = D / 16;  // k-steps of S^T = K Q^T
  constexpr int kMT = D / 16;  // m-tiles of O^T = V^T P^T
  constexpr bool kQReg = kNH * kKS <= 8;  // Q^T fragments kept in registers
  extern __shared__ __align__(16) unsigned char smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, s = blockIdx.z;

  const int len = LDX(p.seq_lens + s);
  const bool bad_len = len < 0 || len > p.seq_cap;
  const int t_begin = split * p.split_len;
  const int t_end = bad_len ? t_begin : min(t_begin + p.split_len, len);
  const int ntile = t_end > t_begin ? (t_end - t_begin + 15) / 16 : 0;
  if (bad_len && threadIdx.x == 0 && split == 0 && h == 0) set_status(p.status, 8u);

  // ---- Q^T fragments (query head 8nh + g of the group, scaled by 2^k into f16) and
  // the per-head score factors, built once by warp 0 into shared memory ----
  uint2* const qfrag = reinterpret_cast<uint2*>(smem);                         // [nh][k-step][32 lanes]
  float* const qfac = reinterpret_cast<float*>(smem + kNH * kKS * 32 * 8);  // [8 kNH heads]
  if (warp == 0) {
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) {
      const int row = 8 * nh + g;
      uint32_t w[D / 8];  // this lane's D/4 dims as bf16 pairs
#pragma unroll
      for (int i = 0; i < D / 8; ++i) w[i] = 0u;
      if (row < p.group) {
        const uint16_t* qp = p.q + static_cast<int64_t>(s) * p.q_row_pitch +
                             static_cast<int64_t>(h * p.group + row) * p.q_head_pitch + c * (D / 4);
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          uint32_t v4[4];
          load16B(qp + 8 * i, v4);
          w[4 * i] = v4[0];
          w[4 * i + 1] = v4[1];
          w[4 * i + 2] = v4[2];
          w[4 * i + 3] = v4[3];
        }
      }
      float am = 0.0f;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) am = fmaxf(am, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
      int k = 0;
      if (am > 0.0f) k = 14 - (static_cast<int>((__float_as_uint(am) >> 23) & 0xFF) - 127);
      k = max(-100, min(120, k));
      const float up = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
      if (c == 0) qfac[row] = p.scale * kLog2e * __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
#pragma unroll
      for (int kb = 0; kb < kKS; ++kb)
        qfrag[(nh * kKS + kb) * 32 + lane] =
            make_uint2(f32x2_to_f16x2(bf16lo(w[2 * kb]) * up, bf16hi(w[2 * kb]) * up),            // dims 4kb, +1
                       f32x2_to_f16x2(bf16lo(w[2 * kb + 1]) * up, bf16hi(w[2 * kb + 1]) * up));  // dims 4kb+2, +3
    }
  }
  __syncthreads();
  float qmul[kNH][2];  // heads 8nh + 2c, + 1
#pragma unroll
  for (int nh = 0; nh < kNH; ++nh) {
    qmul[nh][0] = qfac[8 * nh + 2 * c];
    qmul[nh][1] = qfac[8 * nh + 2 * c + 1];
  }
  uint2 qreg[kQReg ? kNH : 1][kQReg ? kKS : 1];
  if constexpr (kQReg) {
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int kb = 0; kb < kKS; ++kb) qreg[nh][kb] = qfrag[(nh * kKS + kb) * 32 + lane];
  }
  auto qb = [&](int nh, int kb) -> uint2 {
    if constexpr (kQReg) {
      return qreg[nh][kb];
    } else {
      return qfrag[(nh * kKS + kb) * 32 + lane];
    }
  };

  // ---- the warp's tiles through its cp.async ring ----
  unsigned char* const ring = smem + T::kQ + warp * T::kStages * T::kBytes;
  bool bad = false;
  // pool row of token (lane & 15) of the warp's tile number `it` (-1 past the end); the
  // block-table load is issued a tile ahead of its copies, so its latency overlaps
  // the current tile's arithmetic
  auto row_of = [&](int it) -> int64_t {
    const int tile = warp + it * kAttnWarps;
    if (tile >= ntile) return -1;
    int t = t_begin + tile * 16 + (lane & 15);
    if (t >= t_end) t = t_end - 1;  // a valid token's address; masked later
    uint32_t bi, bo;
    p.div_bs.divmod(static_cast<uint32_t>(t), bi, bo);
    int64_t blk = LDX(p.block_table + static_cast<int64_t>(s) * p.max_blocks + bi);
    if (blk < 0 || blk >= p.num_blocks) {
      bad = true;
      blk = 0;
    }
    return (blk * p.block_size + bo) * p.H + h;
  };
  // copies of a tile (rows from row_of, uniform -1 when there is none) into stage st:
  // the 32 lanes take consecutive 16-byte pieces of the 16 rows (whole sectors), then
  // lanes 0-15 the K block and row scales and lanes 16-31 the V ones
  auto issue = [&](int64_t row, int st) {
    if (__shfl_sync(0xFFFFFFFFu, row, 0) < 0) return;
    unsigned char* const sb = ring + st * T::kBytes;
    const int tt = lane & 15;
    constexpr int kPK = T::kCK / 16, kPV = T::kCV / 16;
    if constexpr (kPK == kPV) {  // the same piece of K and V: one row exchange for both
#pragma unroll
      for (int i = lane; i < 16 * kPK; i += 32) {
        const int64_t rr = shfl64(row, i / kPK);
        cp_async16(sb + T::kOffKC + (i / kPK) * T::kSK + (i % kPK) * 16, p.k.codes + rr * T::kCK + (i % kPK) * 16);
        cp_async16(sb + T::kOffVC + (i / kPV) * T::kSV + (i % kPV) * 16, p.v.codes + rr * T::kCV + (i % kPV) * 16);
      }
    } else {
#pragma unroll
      for (int i = lane; i < 16 * kPK; i += 32) {
        const int64_t rr = shfl64(row, i / kPK);
        cp_async16(sb + T::kOffKC + (i / kPK) * T::kSK + (i % kPK) * 16, p.k.codes + rr * T::kCK + (i % kPK) * 16);
      }
#pragma unroll
      for (int i = lane; i < 16 * kPV; i += 32) {
        const int64_t rr = shfl64(row, i / kPV);
        cp_async16(sb + T::kOffVC + (i / kPV) * T::kSV + (i % kPV) * 16, p.v.codes + rr * T::kCV + (i % kPV) * 16);
      }
    }
    if (lane < 16) {
      if constexpr (T::kBK > 0) cp_async_n<T::kBK>(sb + T::kOffKB + tt * T::kBK, p.k.bscale + row * T::kBK);
      cp_async_small<4>(sb + T::kOffKR + tt * 4, p.k.rscale + row);
    } else {
      if constexpr (T::kBV > 0) cp_async_n<T::kBV>(sb + T::kOffVB + tt * T::kBV, p.v.bscale + row * T::kBV);
      cp_async_small<4>(sb + T::kOffVR + tt * 4, p.v.rscale + row);
    }
  };

  AttnState<D, kNH> st;
  st.init();

#pragma unroll
  for (int j = 0; j < T::kStages - 1; ++j) {
    issue(row_of(j), j);
    cp_async_commit();
  }
  const int my_tiles = ntile > warp ? (ntile - warp + kAttnWarps - 1) / kAttnWarps : 0;
  for (int it = 0; it < my_tiles; ++it) {
    const int64_t row_next = row_of(it + T::kStages - 1);  // the refill's rows, loaded early
    cp_async_wait<T::kStages - 2>();
    __syncwarp();
    const unsigned char* const sb = ring + (it % T::kStages) * T::kBytes;
    const int t0 = t_begin + (warp + it * kAttnWarps) * 16;

    const TileView tv{sb + T::kOffKC, sb + T::kOffVC, sb + T::kOffKB, sb + T::kOffVB, sb + T::kOffKR, sb + T::kOffVR,
                      T::kSK, T::kSV, T::kBK, T::kBV, 4};
    attn_tile<D, kFK, kFV, kNH>(tv, qb, qmul, lane, t_end - t0, st);
    __syncwarp();  // every lane has read this stage before it is refilled
    issue(row_next, (it + T::kStages - 1) % T::kStages);
    cp_async_commit();
  }
  cp_async_wait<0>();
  // the merge kernel (when the sequence is split) may be scheduled from here on; it
  // waits for this grid's writes before it reads them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_status(p.status, 2u);
  // row sums over the 8 lanes (tokens) of each head
#pragma unroll
  for (int off = 4; off <= 16; off <<= 1)
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh) {
      st.l[nh][0] += __shfl_xor_sync(0xFFFFFFFFu, st.l[nh][0], off);
      st.l[nh][1] += __shfl_xor_sync(0xFFFFFFFFu, st.l[nh][1], off);
    }
  const bool cta_bad = __syncthreads_or(bad ? 1 : 0) != 0 || bad_len;  // the ring is free after this

  // per warp: O (true scale: O * R) by head and natural dim, and m, l per head
  constexpr int kHeads = 8 * kNH;
  float* const mo = reinterpret_cast<float*>(smem + T::kQ) + warp * kHeads * (D + 2);
#pragma unroll
  for (int q = 0; q < kMT; ++q)
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int head = 8 * nh + 2 * c + (e & 1);
        const int d = g * (D / 8) + 2 * q + (e >> 1);
        mo[head * (D + 2) + d] = st.o[q][nh][e] * st.R;
      }
  if (g == 0) {
#pragma unroll
    for (int nh = 0; nh < kNH; ++nh)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int head = 8 * nh + 2 * c + e;
        mo[head * (D + 2) + D] = st.m[nh][e];
        mo[head * (D + 2) + D + 1] = st.l[nh][e];
      }
  }
  __syncthreads();
  const float* const mall = reinterpret_cast<const float*>(smem + T::kQ);
  for (int idx = threadIdx.x; idx < p.group * D; idx += kAttnThreads) {
    const int row = idx / D, d = idx % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mall[(w * kHeads + row) * (D + 2) + D]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float mw = mall[(w * kHeads + row) * (D + 2) + D];
      const float f = mw == kNegInf ? 0.0f : ex2(mw - M);
      L += mall[(w * kHeads + row) * (D + 2) + D + 1] * f;
      O += mall[(w * kHeads + row) * (D + 2) + d] * f;
    }
    const int qh = h * p.group + row;
    if (p.nsplit == 1) {
      if (cta_bad) continue;  // a bad sequence leaves its output untouched
      const float y = L > 0.0f ? O / L : 0.0f;
      STX(p.out + static_cast<int64_t>(s) * p.o_row_pitch + static_cast<int64_t>(qh) * p.o_head_pitch + d,
          static_cast<uint16_t>(pack_bf16x2(y, 0.0f) & 0xFFFFu));
    } else {
      float* const wsr = p.ws + ((static_cast<int64_t>(s) * p.Hq + qh) * p.nsplit + split) * (D + 2);
      STX(wsr + d, O);
      if (d == 0) {
        STX(wsr + D, M);
        STX(wsr + D + 1, cta_bad ? __int_as_float(0x7FC00000) : L);  // NaN marks a bad sequence
      }
    }
  }
}

// Merge of the splits of each (sequence, query head): o = sum_k O_k 2^(M_k - M) /
// sum_k L_k 2^(M_k - M), one warp per (sequence, query head).  Lane k holds split k's
// M and L (32 splits at a time), the warp reduces them, and each lane sums its D/32
// dims over the splits.  The O rows of the first kPre splits are loaded together with
// M and L, so a call with up to kPre splits waits for memory once.  A NaN L (bad
// sequence) leaves the output untouched.
constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) decode_attn_merge_kernel(const AttnParams p) {
  constexpr int kDL = D / 32 > 0 ? D / 32 : 1;  // dims per lane (D >= 64: 2, 4 or 8)
  constexpr int kPre = 64 / kDL;               // splits whose O is loaded up front
  // launched as a programmatic dependent of the attention kernel: wait for its results
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int sq = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);  // s * Hq + qh
  if (sq >= p.S * p.Hq) return;
  const int s = sq / p.Hq, qh = sq % p.Hq;
  const float* const base = p.ws + static_cast<int64_t>(sq) * p.nsplit * (D + 2);
  const int npre = min(p.nsplit, kPre);
  float2 pre[kPre][kDL / 2];
#pragma unroll
  for (int k = 0; k < kPre; ++k)
#pragma unroll
    for (int i = 0; i < kDL / 2; ++i)
      pre[k][i] = k < npre ? LDX(reinterpret_cast<const float2*>(base + k * (D + 2) + kDL * lane + 2 * i))
                           : make_float2(0.0f, 0.0f);  // (D + 2) * 4 bytes is a multiple of 8
  float M = kNegInf;
  bool bad = false;
  for (int k0 = 0; k0 < p.nsplit; k0 += 32) {
    const int k = k0 + lane;
    if (k < p.nsplit) {
      M = fmaxf(M, LDX(base + k * (D + 2) + D));
      bad = bad || isnan(LDX(base + k * (D + 2) + D + 1));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  if (__any_sync(0xFFFFFFFFu, bad)) return;
  float L = 0.0f;
  float o[kDL];
#pragma unroll
  for (int i = 0; i < kDL; ++i) o[i] = 0.0f;
  for (int k0 = 0; k0 < p.nsplit; k0 += 32) {
    float f = 0.0f;
    const int kk = k0 + lane;
    if (kk < p.nsplit) {
      const float mk = LDX(base + kk * (D + 2) + D);
      f = mk == kNegInf ? 0.0f : ex2(mk - M);
      L += LDX(base + kk * (D + 2) + D + 1) * f;
    }
    if (k0 == 0) {
#pragma unroll
      for (int k = 0; k < kPre; ++k) {
        const float fk = __shfl_sync(0xFFFFFFFFu, f, k);  // 0 past the last split
#pragma unroll
        for (int i = 0; i < kDL / 2; ++i) {
          o[2 * i] += pre[k][i].x * fk;
          o[2 * i + 1] += pre[k][i].y * fk;
        }
      }
    }
    const int kfirst = k0 == 0 ? kPre : 0;
    const int nk = min(32, p.nsplit - k0);
#pragma unroll 4
    for (int k = kfirst; k < nk; ++k) {
      const float fk = __shfl_sync(0xFFFFFFFFu, f, k);
      const float* const ok = base + (k0 + k) * (D + 2) + kDL * lane;
#pragma unroll
      for (int i = 0; i < kDL; i += 2) {
        const float2 v = LDX(reinterpret_cast<const float2*>(ok + i));
        o[i] += v.x * fk;
        o[i + 1] += v.y * fk;
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, off);
  uint16_t* const out = p.out + static_cast<int64_t>(s) * p.o_row_pitch + static_cast<int64_t>(qh) * p.o_head_pitch;
#pragma unroll
  for (int i = 0; i < kDL; i += 2) {
    const float y0 = L > 0.0f ? o[i] / L : 0.0f;
    const float y1 = L > 0.0f ? o[i + 1] / L : 0.0f;
    STX(reinterpret_cast<uint32_t*>(out + kDL * lane + i), pack_bf16x2(y0, y1));
  }
}

// ---------------------------------------------------------------------------------
// Page-major decode attention: one block per (token split, sequence) that covers every
// KV head.  16 consecutive tokens of a page (block_size a multiple of 16) hold, for all
// H heads, one contiguous range of each pool plane: H x 16 code rows, block-scale rows
// and row scales.  So a producer warp moves a stage of P = W / H such 16-token chunks
// with 6 P bulk copies (cp.async.bulk, completion on the stage's "full" mbarrier), and
// W consumer warps each take one (chunk, head) of every stage: warp w serves head w % H
// and chunk w / H, with the tile arithmetic of the head-major kernel above.  A consumer
// releases a stage on its "empty" mbarrier (W arrivals) before the producer refills it.
// Warps of one head (P > 1) merge through shared memory at the end; each head's result
// (or split partial) is written by its chunk-0 warp.
// ---------------------------------------------------------------------------------
template <int D, int kFK, int kFV, int W>
struct PageStage {
  static constexpr int kCK = kFK == 3 ? D : D / 2;
  static constexpr int kCV = kFV == 3 ? D : D / 2;
  static constexpr int kBK = kFK == 3 ? 0 : D / 16;
  static constexpr int kBV = kFV == 3 ? 0 : D / 16;
  static constexpr int kRow = kCK + kCV + kBK + kBV + 8;  // pool bytes per (token, KV head)
  // a stage: 16 W (token, head) rows of every plane; chunk j's rows start at 16 H j
  static constexpr int kOffKC = 0;
  static constexpr int kOffVC = kOffKC + 16 * W * kCK;
  static constexpr int kOffKB = kOffVC + 16 * W * kCV;
  static constexpr int kOffVB = kOffKB + 16 * W * kBK;
  static constexpr int kOffKR = kOffVB + 16 * W * kBV;
  static constexpr int kOffVR = kOffKR + 16 * W * 4;
  static constexpr int kBytes = kOffVR + 16 * W * 4;
  // 2 blocks per SM at W = 8, 1 at W = 16
  static constexpr int kBudget = W == 8 ? 108 * 1024 : 216 * 1024;
  static constexpr int kStagesFit = kBudget / kBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : (kStagesFit < 2 ? 2 : kStagesFit);
  static constexpr int kRing = kStages * kBytes;
  // end-of-block merge: per consumer warp and lane, O (D/16 m-tiles x 4) + m, l (2 each)
  static constexpr int kLaneFloats = (D / 16) * 4 + 4;
  static constexpr int kMerge = W * 32 * kLaneFloats * 4;
  static constexpr int kOffBar = kRing > kMerge ? kRing : kMerge;
  static constexpr int kSmem = kOffBar + 2 * kStages * 8 + 16;  // full + empty barriers, the bad flag
};

template <int D, int kFK, int kFV, int W, int H>
__global__ void __launch_bounds__((W + 1) * 32, W == 8 ? 2 : 1) decode_attn_page_kernel(const AttnParams p) {
  using T = PageStage<D, kFK, kFV, W>;
  constexpr int kKS = D / 16;
  constexpr int kMT = D / 16;
  static_assert(kKS <= 8, "Q^T fragments of one head n-tile in registers");
  extern __shared__ __align__(128) unsigned char page_smem[];
  unsigned char* const smem = page_smem;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int split = blockIdx.x, s = blockIdx.z;
  constexpr int P = W / H;  // 16-token chunks per stage (the KV head count H is fixed per instance)

  const int len = LDX(p.seq_lens + s);
  const bool bad_len = len < 0 || len > p.seq_cap;
  const int t_begin = split * p.split_len;
  const int t_end = bad_len ? t_begin : min(t_begin + p.split_len, len);
  const int nstage = t_end > t_begin ? (t_end - t_begin + 16 * P - 1) / (16 * P) : 0;
  if (bad_len && threadIdx.x == 0 && split == 0) set_status(p.status, 8u);

  const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const uint32_t full0 = ring_s + T::kOffBar;          // full[st] at full0 + 8 st
  const uint32_t empty0 = full0 + 8 * T::kStages;      // empty[st] at empty0 + 8 st
  int* const bad_flag = reinterpret_cast<int*>(smem + T::kOffBar + 16 * T::kStages);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < T::kStages; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, W);
    }
    *bad_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == W) {
    // ---- producer: lane j < P resolves chunk j of each stage and issues its copies ----
    bool timed_out = false, bad = false;
    for (int k = 0; k < nstage; ++k) {
      const int st = k % T::kStages;
      const int t0 = t_begin + 16 * (P * k + lane);
      bool have = false;
      int64_t r0 = 0;  // pool row (slot, head 0) of the chunk's first token
      if (lane < P && t0 < t_end) {
        uint32_t bi, bo;
        p.div_bs.divmod(static_cast<uint32_t>(t0), bi, bo);
        const int64_t blk = LDX(p.block_table + static_cast<int64_t>(s) * p.max_blocks + bi);
        if (blk < 0 || blk >= p.num_blocks) {
          bad = true;
        } else {
          have = true;
          r0 = (blk * p.block_size + bo) * H;
        }
      }
      const uint32_t bytes = __reduce_add_sync(0xFFFFFFFFu, have ? 16u * H * T::kRow : 0u);
      const bool any_bad = __any_sync(0xFFFFFFFFu, bad);
      if (k >= T::kStages && !mbar_wait(empty0 + 8 * st, ((k / T::kStages) - 1) & 1)) timed_out = true;
      if (lane == 0) {
        if (any_bad) *bad_flag = 1;  // published by the arrival below
        mbar_arrive_expect_tx(full0 + 8 * st, bytes);
      }
      __syncwarp();
      if (have) {
        const uint32_t sb = ring_s + st * T::kBytes;
        const int jr = 16 * H * lane;  // the chunk's first row in the stage planes
        const uint32_t full = full0 + 8 * st;
        bulk_copy_g2s(sb + T::kOffKC + jr * T::kCK, p.k.codes + r0 * T::kCK, 16u * H * T::kCK, full);
        bulk_copy_g2s(sb + T::kOffVC + jr * T::kCV, p.v.codes + r0 * T::kCV, 16u * H * T::kCV, full);
        if constexpr (T::kBK > 0) bulk_copy_g2s(sb + T::kOffKB + jr * T::kBK, p.k.bscale + r0 * T::kBK, 16u * H * T::kBK, full);
        if constexpr (T::kBV > 0) bulk_copy_g2s(sb + T::kOffVB + jr * T::kBV, p.v.bscale + r0 * T::kBV, 16u * H * T::kBV, full);
        bulk_copy_g2s(sb + T::kOffKR + jr * 4, p.k.rscale + r0, 16u * H * 4, full);
        bulk_copy_g2s(sb + T::kOffVR + jr * 4, p.v.rscale + r0, 16u * H * 4, full);
      }
    }
    const bool bad_any = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      if (bad_any) set_status(p.status, 2u);
      if (timed_out) set_status(p.status, 16u);
    }
    return;  // the consumers' own barrier below leaves this warp out
  }

  // ---- consumers: warp w serves head h = w % H, chunk j = w / H of every stage ----
  const int h = warp % H, j = warp / H;
  // Q^T fragments (query head h * group + g, this lane's dims c*D/4 + 4kb .. + 3, scaled
  // by a power of two into f16 exactly) and the per-head query factors
  uint2 qreg[kKS];
  float qfac = 0.0f;
  {
    uint32_t w[D / 8];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) w[i] = 0u;
    if (g < p.group) {
      const uint16_t* qp = p.q + static_cast<int64_t>(s) * p.q_row_pitch +
                           static_cast<int64_t>(h * p.group + g) * p.q_head_pitch + c * (D / 4);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t v4[4];
        load16B(qp + 8 * i, v4);
        w[4 * i] = v4[0];
        w[4 * i + 1] = v4[1];
        w[4 * i + 2] = v4[2];
        w[4 * i + 3] = v4[3];
      }
    }
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) am = fmaxf(am, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
    int kq = 0;
    if (am > 0.0f) kq = 14 - (static_cast<int>((__float_as_uint(am) >> 23) & 0xFF) - 127);
    kq = max(-100, min(120, kq));
    const float up = __uint_as_float(static_cast<uint32_t>(127 + kq) << 23);
    qfac = p.scale * kLog2e * __uint_as_float(static_cast<uint32_t>(127 - kq) << 23);
#pragma unroll
    for (int kb = 0; kb < kKS; ++kb)
      qreg[kb] = make_uint2(f32x2_to_f16x2(bf16lo(w[2 * kb]) * up, bf16hi(w[2 * kb]) * up),
                            f32x2_to_f16x2(bf16lo(w[2 * kb + 1]) * up, bf16hi(w[2 * kb + 1]) * up));
  }
  float qmul[1][2];  // heads 2c, 2c + 1: the factors of lanes (2c, 0) and (2c + 1, 0)
  qmul[0][0] = __shfl_sync(0xFFFFFFFFu, qfac, 8 * c);
  qmul[0][1] = __shfl_sync(0xFFFFFFFFu, qfac, 8 * c + 4);
  auto qb = [&](int, int kb) -> uint2 { return qreg[kb]; };

  AttnState<D, 1> st;
  st.init();
  bool timed_out = false;
  for (int k = 0; k < nstage; ++k) {
    const int stg = k % T::kStages;
    if (!mbar_wait(full0 + 8 * stg, (k / T::kStages) & 1)) timed_out = true;
    const int t0 = t_begin + 16 * (P * k + j);
    if (t0 < t_end) {
      const unsigned char* const sb = smem + stg * T::kBytes;
      const int r = 16 * H * j + h;  // row of this chunk's token 0, head h; tokens H rows apart
      const TileView tv{sb + T::kOffKC + r * T::kCK, sb + T::kOffVC + r * T::kCV, sb + T::kOffKB + r * T::kBK,
                        sb + T::kOffVB + r * T::kBV, sb + T::kOffKR + r * 4, sb + T::kOffVR + r * 4,
                        H * T::kCK, H * T::kCV, H * T::kBK, H * T::kBV, H * 4};
      attn_tile<D, kFK, kFV, 1>(tv, qb, qmul, lane, t_end - t0, st);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stg);
  }
  // the merge kernel (when the sequence is split) may be scheduled from here on; it
  // waits for this grid's writes before it reads them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // row sums over the 8 lanes (tokens) of each head
#pragma unroll
  for (int off = 4; off <= 16; off <<= 1) {
    st.l[0][0] += __shfl_xor_sync(0xFFFFFFFFu, st.l[0][0], off);
    st.l[0][1] += __shfl_xor_sync(0xFFFFFFFFu, st.l[0][1], off);
  }
  if (__any_sync(0xFFFFFFFFu, timed_out) && lane == 0) set_status(p.status, 16u);
  // the producer's bad flag is visible: it was set before the arrival of a stage this
  // warp has waited for (or nothing was issued, and it is still 0)
  const bool cta_bad = bad_len || *bad_flag != 0;

  // this lane's O (true scale O * R), m and l for heads 2c, 2c + 1
  float O[kMT][4], M[2], L[2];
#pragma unroll
  for (int q = 0; q < kMT; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) O[q][e] = st.o[q][0][e] * st.R;
  M[0] = st.m[0][0];
  M[1] = st.m[0][1];
  L[0] = st.l[0][0];
  L[1] = st.l[0][1];
  if (P > 1) {
    // the P warps of a head merge through shared memory (the ring is free once every
    // consumer has waited for every stage): warp w's lane values at [w][lane][.]
    asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
    float* const mine = reinterpret_cast<float*>(smem) + (warp * 32 + lane) * T::kLaneFloats;
#pragma unroll
    for (int q = 0; q < kMT; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) mine[4 * q + e] = O[q][e];
    mine[4 * kMT] = M[0];
    mine[4 * kMT + 1] = M[1];
    mine[4 * kMT + 2] = L[0];
    mine[4 * kMT + 3] = L[1];
    asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
    if (j != 0) return;
    const float* const all = reinterpret_cast<const float*>(smem);
    float Mn[2] = {M[0], M[1]};
    for (int jj = 1; jj < P; ++jj) {
      const float* const o = all + ((jj * H + h) * 32 + lane) * T::kLaneFloats;
      Mn[0] = fmaxf(Mn[0], o[4 * kMT]);
      Mn[1] = fmaxf(Mn[1], o[4 * kMT + 1]);
    }
    float f[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      f[e] = M[e] == kNegInf ? 0.0f : ex2(M[e] - Mn[e]);
      L[e] *= f[e];
    }
#pragma unroll
    for (int q = 0; q < kMT; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[q][e] *= f[e & 1];
    for (int jj = 1; jj < P; ++jj) {
      const float* const o = all + ((jj * H + h) * 32 + lane) * T::kLaneFloats;
      float fj[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float mj = o[4 * kMT + e];
        fj[e] = mj == kNegInf ? 0.0f : ex2(mj - Mn[e]);
        L[e] += o[4 * kMT + 2 + e] * fj[e];
      }
#pragma unroll
      for (int q = 0; q < kMT; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[q][e] += o[4 * q + e] * fj[e & 1];
    }
    M[0] = Mn[0];
    M[1] = Mn[1];
  }
  // heads 2c + e (e = 0, 1) of this KV head's group; dims g*D/8 + 2q and + 1
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int head = 2 * c + e;
    if (head >= p.group) continue;
    const int qh = h * p.group + head;
    if (p.nsplit == 1) {
      if (cta_bad) continue;  // a bad sequence leaves its output untouched
      uint16_t* const out = p.out + static_cast<int64_t>(s) * p.o_row_pitch + static_cast<int64_t>(qh) * p.o_head_pitch;
#pragma unroll
      for (int q = 0; q < kMT; ++q) {
        const int d = g * (D / 8) + 2 * q;
        const float y0 = L[e] > 0.0f ? O[q][e] / L[e] : 0.0f;
        const float y1 = L[e] > 0.0f ? O[q][e + 2] / L[e] : 0.0f;
        STX(reinterpret_cast<uint32_t*>(out + d), pack_bf16x2(y0, y1));
      }
    } else {
      float* const wsr = p.ws + ((static_cast<int64_t>(s) * p.Hq + qh) * p.nsplit + split) * (D + 2);
#pragma unroll
      for (int q = 0; q < kMT; ++q) {
        const int d = g * (D / 8) + 2 * q;
        STX(wsr + d, O[q][e]);
        STX(wsr + d + 1, O[q][e + 2]);
      }
      if (g == 0) {
        STX(wsr + D, M[e]);
        STX(wsr + D + 1, cta_bad ? __int_as_float(0x7FC00000) : L[e]);  // NaN marks a bad sequence
      }
    }
  }
}

// The merge as a programmatic dependent launch: it may be scheduled while the attention
// kernel drains and waits (griddepcontrol.wait) for that kernel's writes.
template <int D>
cudaError_t launch_merge(const AttnParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.S * p.Hq + kMergeWarps - 1) / kMergeWarps);
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_attn_merge_kernel<D>, p);
}

template <int D, int kFK, int kFV, int kNH>
cudaError_t attn_launch(const AttnParams& p, cudaStream_t s) {
  using T = AttnTile<D, kFK, kFV>;
  auto k = decode_attn_kernel<D, kFK, kFV, kNH>;
  if (T::kSmem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaSuccess;
  const dim3 grid(p.nsplit, p.H, p.S);
  KVQ_LAUNCH("decode_attn_kernel", s, k<<<grid, kAttnThreads, T::kSmem, s>>>(p); e = cudaGetLastError());
  if (e != cudaSuccess || p.nsplit == 1) return e;
  KVQ_LAUNCH("decode_attn_merge_kernel", s, e = launch_merge<D>(p, s));
  return e;
}

template <int D, int kNH>
cudaError_t attn_dispatch_fmt(const AttnParams& p, cudaStream_t s) {
  const bool k8 = p.fmt_k == 3, v8 = p.fmt_v == 3;
  if (!k8 && !v8) return attn_launch<D, 1, 1, kNH>(p, s);
  if (k8 && !v8) return attn_launch<D, 3, 1, kNH>(p, s);
  if (!k8 && v8) return attn_launch<D, 1, 3, kNH>(p, s);
  return attn_launch<D, 3, 3, kNH>(p, s);
}

// Query heads per KV head: one n-tile of 8 heads, or two for 9 to 16.
template <int D>
cudaError_t attn_dispatch_group(const AttnParams& p, cudaStream_t s) {
  return p.group <= 8 ? attn_dispatch_fmt<D, 1>(p, s) : attn_dispatch_fmt<D, 2>(p, s);
}

template <int D, int kFK, int kFV, int W, int H>
cudaError_t page_launch(const AttnParams& p, cudaStream_t s) {
  using T = PageStage<D, kFK, kFV, W>;
  auto k = decode_attn_page_kernel<D, kFK, kFV, W, H>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nsplit, 1, p.S);
  KVQ_LAUNCH("decode_attn_page_kernel", s, k<<<grid, (W + 1) * 32, T::kSmem, s>>>(p); e = cudaGetLastError());
  if (e != cudaSuccess || p.nsplit == 1) return e;
  KVQ_LAUNCH("decode_attn_merge_kernel", s, e = launch_merge<D>(p, s));
  return e;
}

template <int D, int W, int H>
cudaError_t page_dispatch_fmt(const AttnParams& p, cudaStream_t s) {
  const bool k8 = p.fmt_k == 3, v8 = p.fmt_v == 3;
  if (!k8 && !v8) return page_launch<D, 1, 1, W, H>(p, s);
  if (k8 && !v8) return page_launch<D, 3, 1, W, H>(p, s);
  if (!k8 && v8) return page_launch<D, 1, 3, W, H>(p, s);
  return page_launch<D, 3, 3, W, H>(p, s);
}

// One instance per KV head count: the stage layout's strides are then constants.
template <int D>
cudaError_t page_dispatch(const AttnParams& p, cudaStream_t s) {
  switch (p.H) {
    case 1: return page_dispatch_fmt<D, 8, 1>(p, s);
    case 2: return page_dispatch_fmt<D, 8, 2>(p, s);
    case 4: return page_dispatch_fmt<D, 8, 4>(p, s);
    case 8: return page_dispatch_fmt<D, 8, 8>(p, s);
    case 16: return page_dispatch_fmt<D, 16, 16>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// Split policy: CTAs resident per SM assumed by the wave count (4 at D <= 128), and
// the most waves a split may create.
constexpr int kAttnCtasPerSm = 4;
constexpr int kAttnMaxWaves = 4;

// Built-in split scratch for kvq_decode_attention_noalloc, for callers that cannot
// allocate device memory: it is part of the library image, so every GPU that loads
// the library holds these 48 MiB until the process exits, and no call allocates.
// One array per device, shared by every call on it: calls that overlap on the GPU
// race on it.  Each call writes every partial it later reads, so nothing in it needs
// clearing between calls.  The policy above keeps S*H*nsplit <= 4 waves = 16 * SMs
// CTAs, so the partials take at most 16 * SMs * 16 query heads * (256 + 2) * 4
// bytes: 40.2 MB on 152 SMs.
constexpr size_t kAttnScratchBytes = size_t{48} << 20;
static __device__ __align__(256) float g_attn_scratch[kAttnScratchBytes / sizeof(float)];

// Host code may not pass g_attn_scratch itself to a kernel: on the host that name is a
// stand-in, not a device address.  The device address is looked up once per device,
// with that device current, on the first call there, and kept.
constexpr int kScratchDevices = 64;
static std::atomic<void*> g_scratch_addr[kScratchDevices];
static std::mutex g_scratch_mu;

cudaError_t attn_builtin_scratch(void** ptr, size_t* bytes) {
  *bytes = kAttnScratchBytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
  void* addr = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr == nullptr) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    addr = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (addr == nullptr) {
      e = cudaGetSymbolAddress(&addr, g_attn_scratch);
      if (e != cudaSuccess || addr == nullptr) {
        cudaGetLastError();  // leave no error behind for the launch check
        return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
      }
      g_scratch_addr[dev].store(addr, std::memory_order_release);
    }
  }
  *ptr = addr;
  return cudaSuccess;
}

size_t attn_builtin_scratch_bytes() { return kAttnScratchBytes; }

int attn_num_splits(int32_t S, int32_t H, int32_t max_seq_len) {
  const int64_t pairs = static_cast<int64_t>(S) * H;
  if (pairs <= 0 || max_seq_len <= 0) return 1;
  const int64_t slots = static_cast<int64_t>(kAttnCtasPerSm) * num_sms();  // CTAs resident at once
  int64_t cap = (max_seq_len + 255) / 256;                                  // >= 256 tokens per split
  const int64_t waves_cap = (kAttnMaxWaves * slots) / pairs;                  // <= kAttnMaxWaves waves
  if (waves_cap < cap) cap = waves_cap;
  if (cap > 64) cap = 64;
  // the split count whose last wave is fullest (least idle CTA time), the smallest on ties
  int best = 1;
  double best_fill = 0.0;
  for (int64_t n = 1; n <= cap; ++n) {
    const int64_t ctas = pairs * n;
    const int64_t waves = (ctas + slots - 1) / slots;
    const double fill = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (fill > best_fill + 0.01) {
      best_fill = fill;
      best = static_cast<int>(n);
    }
  }
  return best;
}

// The page-major kernel serves pages of whole 16-token chunks (block_size a multiple of
// 16), head_dim 64 or 128, up to 8 query heads per KV head, and H in {1, 2, 4, 8, 16}
// (W = 8 consumer warps, or 16 at H = 16, P = W / H chunks per stage).
bool attn_page_ok(int32_t block_size, int32_t H, int32_t D, int32_t group) {
  return block_size % 16 == 0 && (D == 64 || D == 128) && group <= 8 &&
         (H == 1 || H == 2 || H == 4 || H == 8 || H == 16);
}

// Splits of the page-major kernel: one block per (split, sequence), 2 resident per SM
// (1 at H = 16); at least 256 tokens a split, and S * H * nsplit <= 16 * SMs so the
// partials stay within the bound of the built-in scratch; the count whose last wave is
// fullest, the smallest on ties.
int attn_page_splits(int32_t S, int32_t H, int32_t max_seq_len) {
  if (S <= 0 || H <= 0 || max_seq_len <= 0) return 1;
  const int64_t slots = static_cast<int64_t>(H == 16 ? 1 : 2) * num_sms();
  int64_t cap = (max_seq_len + 255) / 256;
  const int64_t scratch_cap = (static_cast<int64_t>(kAttnCtasPerSm) * kAttnMaxWaves * num_sms()) /
                              (static_cast<int64_t>(S) * H);
  if (scratch_cap < cap) cap = scratch_cap;
  if (cap > 64) cap = 64;
  int best = 1;
  double best_fill = 0.0;
  for (int64_t n = 1; n <= cap; ++n) {
    const int64_t ctas = static_cast<int64_t>(S) * n;
    const int64_t waves = (ctas + slots - 1) / slots;
    const double fill = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (fill > best_fill + 0.01) {
      best_fill = fill;
      best = static_cast<int>(n);
    }
  }
  return best;
}

// Tokens per split: the splits cover max_seq_len in multiples of `unit` tokens.
static int attn_split_len(int32_t max_seq_len, int nsplit, int unit) {
  const int64_t per = (static_cast<int64_t>(max_seq_len) + nsplit - 1) / nsplit;
  const int64_t len = ((per + unit - 1) / unit) * unit;
  return len > 0 ? static_cast<int>(len) : unit;
}

size_t attn_workspace_bytes(int32_t S, int32_t H, int32_t Hq, int32_t D, int32_t max_seq_len) {
  if (S <= 0 || H <= 0 || Hq <= 0 || D <= 0 || max_seq_len <= 0) return 0;
  // either kernel may serve the call (the choice also depends on the pool's block size)
  int n = attn_num_splits(S, H, max_seq_len);
  const int np = attn_page_splits(S, H, max_seq_len);
  if (np > n) n = np;
  if (n <= 1) return 0;
  return static_cast<size_t>(S) * Hq * n * (D + 2) * sizeof(float);
}

cudaError_t launch_decode_attention(const AttnParams& p_in, cudaStream_t s) {
  AttnParams p = p_in;
  if (attn_page_ok(p.block_size, p.H, p.D, p.group)) {
    p.nsplit = attn_page_splits(p.S, p.H, p.max_len);
    p.split_len = attn_split_len(p.max_len, p.nsplit, 16);
    switch (p.D) {
      case 64: return page_dispatch<64>(p, s);
      case 128: return page_dispatch<128>(p, s);
    }
    return cudaErrorInvalidValue;
  }
  p.nsplit = attn_num_splits(p.S, p.H, p.max_len);
  p.split_len = attn_split_len(p.max_len, p.nsplit, 64);
  switch (p.D) {
    case 64: return attn_dispatch_group<64>(p, s);
    case 128: return attn_dispatch_group<128>(p, s);
    case 256: return attn_dispatch_group<256>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
