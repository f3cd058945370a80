// kvq_device.cuh -- device helpers shared by the codec kernels (sm_103a).
//
// Rounding contract: every floating-point step below is a single IEEE binary32
// operation with round-to-nearest-even, written with the __f*_rn intrinsics so
// that nvcc can neither contract a mul and an add into an FMA nor reorder them.
// Denormals are kept (no -ftz, no fast math).  The FP4/FP8 conversions are the
// hardware cvt instructions (.rn = nearest even, .satfinite = clamp to the
// largest finite value); the tests check them code by code against the oracle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// ---------------------------------------------------------------------------
// checked build (-DKVQ_CHECKED, a debugging aid, never the product library):
// every global access is tested against the byte ranges the host registered for
// the launch and against its alignment; a bad access is counted, the first one
// recorded, and the access skipped.  Each translation unit has its own copy of
// these symbols, set by that unit's launchers.
// ---------------------------------------------------------------------------
#ifdef KVQ_CHECKED
namespace dbg {
struct Range {
  unsigned long long lo, hi;
};
static __device__ Range g_ranges[32];
static __device__ int g_nranges;
static __device__ unsigned long long g_bad[4];  // count, first address, bytes, line

__device__ __forceinline__ bool ok(const void* p, unsigned bytes, unsigned align, unsigned line) {
  const unsigned long long a = reinterpret_cast<unsigned long long>(p);
  bool good = (a % align) == 0;
  if (good) {
    good = false;
    for (int i = 0; i < g_nranges; ++i)
      if (a >= g_ranges[i].lo && a + bytes <= g_ranges[i].hi) {
        good = true;
        break;
      }
  }
  if (!good && atomicAdd(&g_bad[0], 1ull) == 0ull) {
    g_bad[1] = a;
    g_bad[2] = bytes;
    g_bad[3] = line;
  }
  return good;
}
}  // namespace dbg
#define KVQ_OK(p, n, a) ::kvq::dbg::ok((p), (n), (a), __LINE__)
}  // namespace kvq
#include <cstdio>
#include "kvq_params.h"
namespace kvq {
namespace dbg {
// Host side, per translation unit: copy the registered ranges before a launch,
// synchronise after it and print what the kernel recorded.
static inline void before() {
  int n = 0;
  HostRange* r = pending(&n);
  Range dr[32];
  for (int i = 0; i < n; ++i) dr[i] = Range{r[i].lo, r[i].hi};
  cudaMemcpyToSymbol(g_ranges, dr, sizeof(Range) * 32);
  cudaMemcpyToSymbol(g_nranges, &n, sizeof(int));
  unsigned long long z[4] = {0, 0, 0, 0};
  cudaMemcpyToSymbol(g_bad, z, sizeof(z));
}
static inline void after(const char* kernel, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  unsigned long long bad[4] = {0, 0, 0, 0};
  if (e == cudaSuccess) cudaMemcpyFromSymbol(bad, g_bad, sizeof(bad));
  int n = 0;
  HostRange* r = pending(&n);
  std::fprintf(stderr, "[kvq checked] %s: sync=%s bad=%llu", kernel, cudaGetErrorString(e), bad[0]);
  if (bad[0]) {
    std::fprintf(stderr, " first=0x%llx bytes=%llu line=%llu", bad[1], bad[2], bad[3]);
    for (int i = 0; i < n; ++i)
      std::fprintf(stderr, " | %s [0x%llx,0x%llx) off=%lld", r[i].name, r[i].lo, r[i].hi,
                   static_cast<long long>(bad[1] - r[i].lo));
  }
  std::fprintf(stderr, "\n");
}
}  // namespace dbg
#else
#define KVQ_OK(p, n, a) true
#endif

#ifdef KVQ_CHECKED
#define KVQ_LAUNCH(name, stream, ...) \
  do {                                \
    ::kvq::dbg::before();             \
    __VA_ARGS__;                      \
    ::kvq::dbg::after(name, stream);  \
  } while (0)
#else
#define KVQ_LAUNCH(name, stream, ...) \
  do {                                \
    __VA_ARGS__;                      \
  } while (0)
#endif

template <typename T>
__device__ __forceinline__ T ldx(const T* p, unsigned line) {
#ifdef KVQ_CHECKED
  if (!dbg::ok(p, sizeof(T), alignof(T), line)) return T{};
#endif
  (void)line;
  return *p;
}
template <typename T>
__device__ __forceinline__ void stx(T* p, T v, unsigned line) {
#ifdef KVQ_CHECKED
  if (!dbg::ok(p, sizeof(T), alignof(T), line)) return;
#endif
  (void)line;
  *p = v;
}
#define LDX(p) ::kvq::ldx((p), __LINE__)
#define STX(p, v) ::kvq::stx((p), (v), __LINE__)

constexpr float kE2M1Max = 6.0f;    // largest E2M1 magnitude
constexpr float kE4M3Max = 448.0f;  // largest finite E4M3 value

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------
// 32 bytes = 16 bf16 = one NVFP4 block, read with one 256-bit load when the
// address is 32-byte aligned (kV8) and with two 128-bit loads otherwise.
// kNC selects the read-only path; it is off where a kernel may write the same
// rows it reads (in-place residual decode).
template <bool kV8, bool kNC>
__device__ __forceinline__ void load32B(const void* p, uint32_t (&w)[8]) {
  if (!KVQ_OK(p, 32, kV8 ? 32 : 16)) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0u;
    return;
  }
  if constexpr (kV8 && kNC) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
          "=r"(w[6]), "=r"(w[7])
        : "l"(p));
  } else if constexpr (kV8) {
    asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p)
                 : "memory");
  } else if constexpr (kNC) {
    const char* c = static_cast<const char*>(p);
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
        : "l"(c));
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
        : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "l"(c + 16));
  } else {
    const char* c = static_cast<const char*>(p);
    asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "l"(c)
                 : "memory");
    asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(c + 16)
                 : "memory");
  }
}

template <bool kV8>
__device__ __forceinline__ void store32B(void* p, const uint32_t (&w)[8]) {
  if (!KVQ_OK(p, 32, kV8 ? 32 : 16)) return;
  if constexpr (kV8) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
    char* c = static_cast<char*>(p);
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(c), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3])
                 : "memory");
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(c + 16), "r"(w[4]), "r"(w[5]),
                 "r"(w[6]), "r"(w[7])
                 : "memory");
  }
}

__device__ __forceinline__ void store8B(void* p, uint32_t a, uint32_t b) {
  if (!KVQ_OK(p, 8, 8)) return;
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void load8B(const void* p, uint32_t& a, uint32_t& b) {
  if (!KVQ_OK(p, 8, 8)) {
    a = b = 0u;
    return;
  }
  asm volatile("ld.global.nc.v2.b32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "l"(p));
}

// ---------------------------------------------------------------------------
// bf16 / fp16 / fp32
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 (lo in bits 0..15), each rounded to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16(a - b) and bf16(a + b) of packed bf16 pairs, each half rounded once to nearest
// even.  For finite bf16 operands this equals the binary32 difference (sum) rounded to
// bf16: the binary32 result is exact when the exponents differ by at most 16, and
// otherwise the smaller operand lies below half a bf16 ulp of the larger, so both
// roundings return the larger (checked for all 4.3e9 pairs of finite bf16 values).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) {
  uint16_t h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}

// Largest |x| of the 16 bf16 in w (returned as fp32).  Comparisons only: exact.
// max.xorsign.abs compares magnitudes; only the sign of its result is
// meaningless, and it is cleared at the end.
__device__ __forceinline__ float absmax16(const uint32_t (&w)[8]) {
  uint32_t m = w[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(w[i]));
  m &= 0x7FFF7FFFu;
  return fmaxf(bf16lo(m), bf16hi(m));
}

// Two fp32 packed in one 64-bit register (lo = element 0).
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo_bits, uint32_t hi_bits) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, uint32_t& lo_bits, uint32_t& hi_bits) {
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo_bits), "=r"(hi_bits) : "l"(v));
}
// Element-wise binary32 product of two pairs, each rounded to nearest even.
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Byte merge: the low byte of each of a, b, c, d into one word (a lowest).
__device__ __forceinline__ uint32_t bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  uint32_t ab, cd, r;
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(ab) : "r"(a), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(cd) : "r"(c), "r"(d));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r) : "r"(ab), "r"(cd));
  return r;
}

// ---------------------------------------------------------------------------
// E4M3 and E2M1
// ---------------------------------------------------------------------------
// Non-negative fp32 -> E4M3 byte, nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_from_f32(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}

// E4M3 byte -> fp16x2 bits (the value in the low half; every E4M3 value is an
// fp16 value, so this is exact).
__device__ __forceinline__ uint32_t e4m3_to_f16x2(uint32_t byte) {
  uint32_t r;
  uint16_t in = static_cast<uint16_t>(byte & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
  return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  return f16_bits_to_f32(static_cast<uint16_t>(e4m3_to_f16x2(byte) & 0xFFFFu));
}

// Two non-negative fp32 -> two E4M3 bytes (lo in bits 0..7, hi in 8..15), nearest
// even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The E4M3 code of the block scale t = min((vb / 6) / rs, 448) (0 when rs == 0),
// exactly as the two divisions define it, usually without dividing.
//
// te = (vb * RN(1/6)) * RN(1/rs) carries four roundings and the defined t two, so
// when every intermediate is a normal binary32 (rs, vb >= 2^-120 ensures it for
// any t near a code boundary) |t / te - 1| <= 6.001 * 2^-24.  The bracket
// [te * (1 - 2^-20), te * (1 + 2^-20)] therefore holds t even after its own
// rounding, and E4M3 rounding is monotone: when both ends of the bracket round to
// the same code, t rounds to it too.  Otherwise (a bracket across a rounding
// boundary, or tiny operands) t is computed by the two divisions.
__device__ __forceinline__ uint32_t block_scale_code(float vb, float rs, float rinv) {
  if (rs >= 0x1p-120f && vb >= 0x1p-120f) {
    const float te = __fmul_rn(__fmul_rn(vb, 0x1.555556p-3f), rinv);
    const float lo = fminf(__fmul_rn(te, 0x1.ffffep-1f), kE4M3Max);
    const float hi = fminf(__fmul_rn(te, 0x1.00001p+0f), kE4M3Max);
    const uint32_t two = e4m3x2_from_f32(lo, hi);
    if ((two & 0xFFu) == (two >> 8)) return two & 0xFFu;
  }
  float t = 0.0f;
  if (rs != 0.0f) t = __fdiv_rn(__fdiv_rn(vb, kE2M1Max), rs);
  return e4m3_from_f32(fminf(t, kE4M3Max));
}

// Mixed-precision exact product: fp32(a_f16) * fp32(b_f16) + (-0), one rounding
// (none here: an E2M1 value times an E4M3 value has at most 6 significant bits).
__device__ __forceinline__ float mul_f16_to_f32(uint16_t a, uint16_t b) {
  float r;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(r) : "h"(a), "h"(b), "f"(-0.0f));
  return r;
}

// Two fp32 -> one byte of E2M1 codes: `lo` in bits 0..3, `hi` in bits 4..7.
// Nearest even, saturating at +-6, sign kept (including -0 and negatives that
// round to zero).
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// One byte of E2M1 codes -> fp16x2 (low nibble -> low half).  Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(r)
      : "r"(byte));
  return r;
}

__device__ __forceinline__ void f16x2_to_f32(uint32_t h2, float& lo, float& hi) {
  lo = f16_bits_to_f32(static_cast<uint16_t>(h2 & 0xFFFFu));
  hi = f16_bits_to_f32(static_cast<uint16_t>(h2 >> 16));
}

// Codes of one 16-element block against s = bs * rs; returns the 8 code bytes as
// two words (low nibble of each byte = the even element).
__device__ __forceinline__ void quantize_block(const uint32_t (&w)[8], float s, uint32_t& c0,
                                               uint32_t& c1) {
  const float inv = (s != 0.0f) ? __frcp_rn(s) : 0.0f;
  uint32_t byte[8];
  if (!isinf(inv)) {
    const uint64_t inv2 = pack_f32x2(__float_as_uint(inv), __float_as_uint(inv));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t ql, qh;
      unpack_f32x2(mul_f32x2(pack_f32x2(w[i] << 16, w[i] & 0xFFFF0000u), inv2), ql, qh);
      byte[i] = e2m1x2_from_f32(__uint_as_float(ql), __uint_as_float(qh));
    }
  } else {  // tiny scale: the reciprocal overflowed, divide directly
#pragma unroll
    for (int i = 0; i < 8; ++i)
      byte[i] = e2m1x2_from_f32(__fdiv_rn(bf16lo(w[i]), s), __fdiv_rn(bf16hi(w[i]), s));
  }
  c0 = bytes4(byte[0], byte[1], byte[2], byte[3]);
  c1 = bytes4(byte[4], byte[5], byte[6], byte[7]);
}

// NVFP4 decode of one 16-element block: y = bf16((e2m1 * bs) * rs).  e2m1 * bs is
// exact (fma.rn.f32.f16 of two fp16 values, at most 6 significant bits), then one
// binary32 rounding by the row scale, then bf16.
__device__ __forceinline__ void nvfp4_decode16(uint32_t cw0, uint32_t cw1, uint32_t bsb, float rs,
                                               uint32_t (&out)[8]) {
  const uint16_t bs16 = static_cast<uint16_t>(e4m3_to_f16x2(bsb) & 0xFFFFu);
  const uint64_t rs2 = pack_f32x2(__float_as_uint(rs), __float_as_uint(rs));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = ((i < 4 ? cw0 : cw1) >> (8 * (i & 3))) & 0xFFu;
    const uint32_t h2 = e2m1x2_to_f16x2(byte);
    const float lo = mul_f16_to_f32(static_cast<uint16_t>(h2 & 0xFFFFu), bs16);
    const float hi = mul_f16_to_f32(static_cast<uint16_t>(h2 >> 16), bs16);
    uint32_t yl, yh;
    unpack_f32x2(mul_f32x2(pack_f32x2(__float_as_uint(lo), __float_as_uint(hi)), rs2), yl, yh);
    out[i] = pack_bf16x2(__uint_as_float(yl), __uint_as_float(yh));
  }
}

// FP8 E4M3 row codec, one 16-element block: q = x * inv (or x / rs when inv is
// infinite), codes E4M3 nearest even, saturating at 448, sign of x; the 16 code
// bytes land in c (element 0 in the low byte of c[0]).
__device__ __forceinline__ void fp8_quantize16(const uint32_t (&w)[8], float rs, float inv,
                                               uint32_t (&c)[4]) {
  c[0] = c[1] = c[2] = c[3] = 0u;
  if (!isinf(inv)) {
    const uint64_t inv2 = pack_f32x2(__float_as_uint(inv), __float_as_uint(inv));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t ql, qh;
      unpack_f32x2(mul_f32x2(pack_f32x2(w[i] << 16, w[i] & 0xFFFF0000u), inv2), ql, qh);
      c[i / 2] |= e4m3x2_from_f32(__uint_as_float(ql), __uint_as_float(qh)) << (16 * (i % 2));
    }
  } else {  // tiny scale: the reciprocal overflowed, divide directly
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i / 2] |= e4m3x2_from_f32(__fdiv_rn(bf16lo(w[i]), rs), __fdiv_rn(bf16hi(w[i]), rs)) << (16 * (i % 2));
  }
}

// FP8 decode of one 16-element block: y = bf16(e4m3 * rs) (E4M3 -> fp16 is exact).
__device__ __forceinline__ void fp8_decode16(const uint32_t (&c)[4], float rs, uint32_t (&out)[8]) {
  const uint64_t rs2 = pack_f32x2(__float_as_uint(rs), __float_as_uint(rs));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t h2;
    const uint16_t two = static_cast<uint16_t>((c[i / 2] >> (16 * (i % 2))) & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    float lo, hi;
    f16x2_to_f32(h2, lo, hi);
    uint32_t yl, yh;
    unpack_f32x2(mul_f32x2(pack_f32x2(__float_as_uint(lo), __float_as_uint(hi)), rs2), yl, yh);
    out[i] = pack_bf16x2(__uint_as_float(yl), __uint_as_float(yh));
  }
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// INT4 decode of 8 codes (one word, low nibble first) with per-element minimum and
// scale: y = bf16(code * sc + mn), a multiply then an add, each rounded (no FMA).
__device__ __forceinline__ void int4_decode8(uint32_t cw, const float (&mn)[8], const float (&sc)[8],
                                             uint32_t (&out)[4]) {
  const uint64_t neg = pack_f32x2(0xCB000000u, 0xCB000000u);  // -2^23
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t byte = (cw >> (8 * i)) & 0xFFu;
    // 2^23 + c is exact for c < 16, so adding -2^23 gives float(c) exactly
    const uint64_t c2 = add_f32x2(pack_f32x2(0x4B000000u | (byte & 15u), 0x4B000000u | (byte >> 4)), neg);
    uint64_t v = mul_f32x2(c2, pack_f32x2(__float_as_uint(sc[2 * i]), __float_as_uint(sc[2 * i + 1])));
    v = add_f32x2(v, pack_f32x2(__float_as_uint(mn[2 * i]), __float_as_uint(mn[2 * i + 1])));
    uint32_t yl, yh;
    unpack_f32x2(v, yl, yh);
    out[i] = pack_bf16x2(__uint_as_float(yl), __uint_as_float(yh));
  }
}

// INT4 decode of 16 codes (8 bytes) with per-element fp32 minimum and scale:
// y = bf16(code * sc + mn), a multiply then an add, each rounded (no FMA).
__device__ __forceinline__ void int4_decode16(uint32_t cw0, uint32_t cw1, const float (&mn)[16],
                                              const float (&sc)[16], uint32_t (&out)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = ((i < 4 ? cw0 : cw1) >> (8 * (i & 3))) & 0xFFu;
    // 2^23 + c is exact for c < 16, so subtracting 2^23 gives float(c) exactly
    uint64_t c2 = pack_f32x2(0x4B000000u | (byte & 15u), 0x4B000000u | (byte >> 4));
    uint64_t neg = pack_f32x2(0xCB000000u, 0xCB000000u);  // -2^23
    c2 = add_f32x2(c2, neg);
    uint64_t v = mul_f32x2(c2, pack_f32x2(__float_as_uint(sc[2 * i]), __float_as_uint(sc[2 * i + 1])));
    v = add_f32x2(v, pack_f32x2(__float_as_uint(mn[2 * i]), __float_as_uint(mn[2 * i + 1])));
    uint32_t yl, yh;
    unpack_f32x2(v, yl, yh);
    out[i] = pack_bf16x2(__uint_as_float(yl), __uint_as_float(yh));
  }
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status != nullptr && KVQ_OK(status, 4, 4)) atomicOr(status, bit);
}

// 16-byte load (four words), read-only path.
__device__ __forceinline__ void load16B(const void* p, uint32_t (&w)[4]) {
  if (!KVQ_OK(p, 16, 16)) {
    w[0] = w[1] = w[2] = w[3] = 0u;
    return;
  }
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p));
}

// 16-byte asynchronous copy global -> shared memory through L2 only (cp.async.cg).
// It lands by the cp.async.wait_group that covers its commit group; the hardware
// tracks it, so no wait in this code spins.  The checked build stores zeros instead
// of copying from outside a registered range.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  if (!KVQ_OK(gsrc, 16, 16)) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
    return;
  }
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// mbarrier objects in shared memory (8 bytes, 8-byte aligned), addressed by their
// 32-bit shared-window address.
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t arrivals) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(arrivals) : "memory");
}
// Makes this thread's initialisations visible to the other threads and to the bulk-copy
// unit; a __syncthreads follows it.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// One arrival that also raises the phase's expected transaction count by `bytes`.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// Tests whether the phase of the given parity has completed; while it has not, the
// thread may be suspended for at most about a microsecond first.
__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(mbar), "r"(parity), "r"(1000u)
      : "memory");
  return done != 0u;
}
// Waits for the phase of the given parity to complete, giving up after a bounded number
// of tries (about 0.1 s); returns whether the phase completed.
constexpr int kMbarTries = 1 << 17;
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
  for (int n = 0; n < kMbarTries; ++n)
    if (mbar_try_wait(mbar, parity)) return true;
  return false;
}
// Bulk copy (cp.async.bulk) of `bytes` bytes (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory; its completion counts `bytes` against the
// current phase of the mbarrier at `mbar`.  The checked build stores zeros, and
// completes the count itself, instead of copying from outside a registered range.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  if (!KVQ_OK(src, bytes, 16)) {
    for (uint32_t o = 0; o < bytes; o += 16)
      asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst + o), "r"(0u) : "memory");
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
    return;
  }
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte load through the coherent path (for rows this launch also writes).
__device__ __forceinline__ void load16B_rw(const void* p, uint32_t (&w)[4]) {
  if (!KVQ_OK(p, 16, 16)) {
    w[0] = w[1] = w[2] = w[3] = 0u;
    return;
  }
  asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p)
               : "memory");
}

__device__ __forceinline__ void store16B(void* p, const uint32_t (&w)[4]) {
  if (!KVQ_OK(p, 16, 16)) return;
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3])
               : "memory");
}

// Width-limited butterfly reductions inside aligned groups of `kWidth` lanes.
template <int kWidth>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = kWidth / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
template <int kWidth>
__device__ __forceinline__ float group_min(float v) {
#pragma unroll
  for (int o = kWidth / 2; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

}  // namespace kvq
