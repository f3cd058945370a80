// payload_kernels.cu -- decode of a logical packed tensor (NVFP4 rows or INT4 groups)
// to bf16, alone (unpack) or added onto a predecessor (residual decode).
//
// Sources: "vllm-rlt PR #166: INT4 KV packing/unpacking and cross-loop residual
// reconstruction", Purpose: unpack_kv(packed); decode_residual(residual, previous)
// with compact sparse rows carrying an int32 position map and absent rows
// inheriting the predecessor.  Arithmetic (binary32, nearest even, no FMA):
//   NVFP4  y = bf16((e2m1 * bs) * rs)
//   INT4   y = bf16(code * fp32(sc16) + fp32(mn16))   (a mul, then an add)
//   residual out[pos[p]] = bf16(prev[pos[p]] + y[p]); other rows keep prev.
//
// Iteration spaces:
//   unpack            every (row, head) of the payload
//   residual in place every kept row: t = pos[p] (the other rows are already prev)
//   residual copy     every row t of out; t is looked up in the sorted pos map by
//                     binary search (kept: add, absent: copy prev)
#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;

// 16 decoded bf16 (packed in w) of payload row p, head h, block b.
template <int kFmt>
__device__ __forceinline__ void decode_block(const UnpackParams& u, int64_t p, int32_t h, int b,
                                             uint32_t (&w)[8]) {
  const PayloadRef& P = u.pay;
  const int64_t prow = p * u.H + h;
  uint32_t cw0, cw1;
  load8B(P.codes + prow * (u.D / 2) + 8 * b, cw0, cw1);
  if constexpr (kFmt == 1) {
    const uint32_t bsb = LDX(static_cast<const uint8_t*>(P.meta0) + prow * u.nb + b);
    const float rs = LDX(P.rscale + prow);
    const uint32_t bs2 = e4m3_to_f16x2(bsb) & 0xFFFFu;
    const uint32_t bsx2 = bs2 | (bs2 << 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = ((i < 4 ? cw0 : cw1) >> (8 * (i & 3))) & 0xFFu;
      float lo, hi;
      f16x2_to_f32(hmul2_bits(e2m1x2_to_f16x2(byte), bsx2), lo, hi);
      w[i] = pack_bf16x2(__fmul_rn(lo, rs), __fmul_rn(hi, rs));
    }
  } else {
    const uint16_t* mnp = static_cast<const uint16_t*>(P.meta0);
    const uint16_t* scp = static_cast<const uint16_t*>(P.meta1);
    float mn[16], sc[16];
    if (P.kind == 0) {  // KEY: per-channel metadata of group p / G
      const int64_t m = ((p / P.G) * u.H + h) * u.D + 16 * b;
      uint32_t a[8], c[8];
      load32B<false, true>(mnp + m, a);
      load32B<false, true>(scp + m, c);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mn[2 * i] = f16_bits_to_f32(static_cast<uint16_t>(a[i] & 0xFFFFu));
        mn[2 * i + 1] = f16_bits_to_f32(static_cast<uint16_t>(a[i] >> 16));
        sc[2 * i] = f16_bits_to_f32(static_cast<uint16_t>(c[i] & 0xFFFFu));
        sc[2 * i + 1] = f16_bits_to_f32(static_cast<uint16_t>(c[i] >> 16));
      }
    } else {  // VALUE: one group covers the whole 16-channel block
      const int ngv = (u.D + P.G - 1) / P.G;
      const int64_t m = prow * ngv + (16 * b) / P.G;
      const float mv = f16_bits_to_f32(LDX(mnp + m));
      const float sv = f16_bits_to_f32(LDX(scp + m));
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        mn[i] = mv;
        sc[i] = sv;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = ((i < 4 ? cw0 : cw1) >> (8 * (i & 3))) & 0xFFu;
      const float lo = __fadd_rn(__fmul_rn(static_cast<float>(byte & 15u), sc[2 * i]), mn[2 * i]);
      const float hi =
          __fadd_rn(__fmul_rn(static_cast<float>(byte >> 4), sc[2 * i + 1]), mn[2 * i + 1]);
      w[i] = pack_bf16x2(lo, hi);
    }
  }
}

__device__ __forceinline__ int32_t find_pos(const int32_t* pos, int32_t n, int32_t t) {
  int32_t lo = 0, hi = n;  // first index with pos[i] >= t
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (LDX(pos + mid) < t)
      lo = mid + 1;
    else
      hi = mid;
  }
  return (lo < n && LDX(pos + lo) == t) ? lo : -1;
}

template <int L, bool kV8, int kFmt, int kMode>
__global__ void __launch_bounds__(kThreads) payload_kernel(const UnpackParams u) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int b = lane % L;
  const int sub = lane / L;
  const uint32_t stride = gridDim.x * (kThreads / 32) * kRowsPerWarp;

  if constexpr (kMode == 2) {  // the copy mode does not visit kept rows by p: check the map here
    if (u.pos != nullptr) {
      for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < u.num_pos;
           i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int32_t ps = LDX(u.pos + i);
        if (ps < 0 || ps >= u.src_rows || (i > 0 && LDX(u.pos + i - 1) >= ps)) set_status(u.status, 4u);
      }
    }
  }
  if (b >= u.nb) return;

  for (uint32_t row = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
       row < u.total_rows; row += stride) {
    uint32_t r, h;
    u.div_h.divmod(row, r, h);
    uint32_t w[8];
    if constexpr (kMode == 0) {
      decode_block<kFmt>(u, r, h, b, w);
      store32B<kV8>(u.y + static_cast<int64_t>(r) * u.y_row_pitch +
                        static_cast<int64_t>(h) * u.y_head_pitch + 16 * b,
                    w);
    } else {
      int64_t t, p;
      if constexpr (kMode == 1) {  // in place: row r is the compact index p
        p = r;
        t = r;
        if (u.pos != nullptr) {
          t = LDX(u.pos + r);
          bool bad = t < 0 || t >= u.src_rows;
          if (h == 0 && b == 0 && r > 0 && LDX(u.pos + r - 1) >= t) set_status(u.status, 4u);
          if (bad) {
            if (h == 0 && b == 0) set_status(u.status, 4u);
            continue;
          }
        }
      } else {  // copy: row r is the output row t
        t = r;
        // both arms signed: a -1 from find_pos must stay negative (with an unsigned
        // arm the conditional would convert it to 0xFFFFFFFF)
        p = (u.pos != nullptr) ? static_cast<int64_t>(find_pos(u.pos, u.num_pos, static_cast<int32_t>(r)))
                               : static_cast<int64_t>(r);
      }
      uint32_t q[8];
      load32B<kV8, kMode == 2>(u.prev + t * u.prev_row_pitch +
                                   static_cast<int64_t>(h) * u.prev_head_pitch + 16 * b,
                               q);
      if (p >= 0) {
        decode_block<kFmt>(u, p, h, b, w);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          q[i] = pack_bf16x2(__fadd_rn(bf16lo(q[i]), bf16lo(w[i])),
                             __fadd_rn(bf16hi(q[i]), bf16hi(w[i])));
      }
      store32B<kV8>(u.y + t * u.y_row_pitch + static_cast<int64_t>(h) * u.y_head_pitch + 16 * b, q);
    }
  }
}

template <int L, bool kV8, int kFmt, int kMode>
cudaError_t pl_launch(const UnpackParams& u, cudaStream_t s) {
  auto k = payload_kernel<L, kV8, kFmt, kMode>;
  int occ = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, 0);
  if (occ < 1) occ = 1;
  const int rows_per_cta = (kThreads / 32) * (32 / L);
  int64_t need = (static_cast<int64_t>(u.total_rows) + rows_per_cta - 1) / rows_per_cta;
  int64_t cap = static_cast<int64_t>(num_sms()) * occ;
  if (need < 1) need = 1;
  const int grid = static_cast<int>(need < cap ? need : cap);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("payload_kernel", s, k<<<grid, kThreads, 0, s>>>(u); e = cudaGetLastError());
  return e;
}

template <int L, bool kV8>
cudaError_t pl_dispatch_fm(const UnpackParams& u, cudaStream_t s) {
  const int f = u.pay.fmt == 1 ? 1 : 2;
  switch (u.mode * 2 + (f - 1)) {
    case 0: return pl_launch<L, kV8, 1, 0>(u, s);
    case 1: return pl_launch<L, kV8, 2, 0>(u, s);
    case 2: return pl_launch<L, kV8, 1, 1>(u, s);
    case 3: return pl_launch<L, kV8, 2, 1>(u, s);
    case 4: return pl_launch<L, kV8, 1, 2>(u, s);
    case 5: return pl_launch<L, kV8, 2, 2>(u, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_payload_decode(const UnpackParams& u, int lanes, bool v8, cudaStream_t s) {
#define KVQ_PL(LN) \
  case LN:         \
    return v8 ? pl_dispatch_fm<LN, true>(u, s) : pl_dispatch_fm<LN, false>(u, s);
  switch (lanes) {
    KVQ_PL(1)
    KVQ_PL(2)
    KVQ_PL(4)
    KVQ_PL(8)
    KVQ_PL(16)
    KVQ_PL(32)
  }
#undef KVQ_PL
  return cudaErrorInvalidValue;
}

}  // namespace kvq
