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
// Work mapping: a lane owns BPL consecutive 16-element blocks of a row (as in the
// NVFP4 kernels).  Iteration spaces:
//   unpack            every (row, head) of the payload, grid-stride
//   residual in place every kept row: t = pos[p] (the other rows are already prev)
//   residual copy     every row t of out, in contiguous runs of tokens per warp (4
//                     to 64, so that short tensors still spread over the GPU): one
//                     binary search of the sorted position map at the start of a run,
//                     then a cursor that only moves forward
// INT4 K unpack (groups over token rows) decodes column-wise instead: see
// int4_key_decode_kernel.  INT4 K residual decodes run row by row here, each row
// reading its group's FP16 minimum and scale per channel.
#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;

// BPL decoded blocks (16 bf16 each, packed in w) of payload row p, head h, from
// block b0 on.
template <int kFmt, int BPL>
__device__ __forceinline__ void decode_blocks(const UnpackParams& u, int64_t p, int32_t h, int b0,
                                              uint32_t (&w)[BPL][8]) {
  const PayloadRef& P = u.pay;
  const int64_t prow = p * u.H + h;
  if constexpr (kFmt == 3) {  // FP8: 16 E4M3 bytes per block, one scale per row
    const float rs = LDX(P.rscale + prow * P.rs_stride);
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      uint32_t c4[4];
      load16B(P.codes + prow * u.D + 16 * (b0 + j), c4);
      fp8_decode16(c4, rs, w[j]);
    }
    return;
  }
  uint32_t cw[2 * BPL];
  if constexpr (BPL == 2) {
    uint32_t c4[4];
    load16B(P.codes + prow * (u.D / 2) + 8 * b0, c4);
#pragma unroll
    for (int i = 0; i < 4; ++i) cw[i] = c4[i];
  } else {
    load8B(P.codes + prow * (u.D / 2) + 8 * b0, cw[0], cw[1]);
  }
  if constexpr (kFmt == 1) {
    const uint8_t* bsp = static_cast<const uint8_t*>(P.meta0) + prow * u.nb + b0;
    uint32_t bsb;
    if constexpr (BPL == 2)
      bsb = LDX(reinterpret_cast<const uint16_t*>(bsp));
    else
      bsb = LDX(bsp);
    const float rs = LDX(P.rscale + prow * P.rs_stride);
#pragma unroll
    for (int j = 0; j < BPL; ++j) nvfp4_decode16(cw[2 * j], cw[2 * j + 1], (bsb >> (8 * j)) & 0xFFu, rs, w[j]);
  } else {
    const uint16_t* mnp = static_cast<const uint16_t*>(P.meta0);
    const uint16_t* scp = static_cast<const uint16_t*>(P.meta1);
    const int gshift = __ffs(P.G) - 1;  // G is a power of two (16 .. 512)
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      const int b = b0 + j;
      float mn[16], sc[16];
      if (P.kind == 0) {  // KEY: per-channel metadata of group p / G
        const int64_t m = ((p >> gshift) * u.H + h) * u.D + 16 * b;  // group p / G
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
        const int ngv = (u.D + P.G - 1) >> gshift;
        const int64_t m = prow * ngv + ((16 * b) >> gshift);
        const float mv = f16_bits_to_f32(LDX(mnp + m));
        const float sv = f16_bits_to_f32(LDX(scp + m));
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          mn[i] = mv;
          sc[i] = sv;
        }
      }
      int4_decode16(cw[2 * j], cw[2 * j + 1], mn, sc, w[j]);
    }
  }
}

// out row = bf16(prev + y) for the BPL blocks of this lane, or a copy of prev when
// `add` is false (kNC: prev is read-only in this launch, i.e. it is not the output).
template <bool kV8, bool kNC, int BPL>
__device__ __forceinline__ void add_store(const uint16_t* prev, uint16_t* out, int b0,
                                          const uint32_t (&w)[BPL][8], bool add) {
#pragma unroll
  for (int j = 0; j < BPL; ++j) {
    uint32_t q[8];
    load32B<kV8, kNC>(prev + 16 * (b0 + j), q);
    if (add) {
#pragma unroll
      for (int i = 0; i < 8; ++i) q[i] = bf16x2_add(q[i], w[j][i]);
    }
    store32B<kV8>(out + 16 * (b0 + j), q);
  }
}

template <int L, int BPL, bool kV8, int kFmt, int kMode>
__global__ void __launch_bounds__(kThreads) payload_kernel(const UnpackParams u) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int li = lane % L;
  const int sub = lane / L;
  const int b0 = li * BPL;
  const uint32_t gwarp = blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
  const uint32_t nwarps = gridDim.x * (kThreads / 32);

  if constexpr (kMode == 2) {  // the copy mode does not visit kept rows by p: check the map here
    if (u.pos != nullptr) {
      for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < u.num_pos;
           i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int32_t ps = LDX(u.pos + i);
        if (ps < 0 || ps >= u.src_rows || (i > 0 && LDX(u.pos + i - 1) >= ps)) set_status(u.status, 4u);
      }
    }
  }
  if constexpr (kMode == 2) {
    // residual decode into a separate output: every row t of out, in runs of u.run <= 32
    // tokens per warp.  The kept tokens of a run come from one read of the position
    // map: a 32-way search finds the first position at or after the run's first token,
    // the 32 lanes read the positions from there, and their OR is the run's bit mask of
    // kept tokens; a kept token's compact index is that first index plus the kept
    // tokens before it.  Lanes without a block of their own join the search and the OR
    // and do nothing else.
    const bool active = b0 < u.nb;
    const uint32_t nruns = (static_cast<uint32_t>(u.src_rows) + u.run - 1) / u.run;
    for (uint32_t run = gwarp; run < nruns; run += nwarps) {
      const int32_t t0 = static_cast<int32_t>(run * u.run);
      const int32_t t1 = min(u.src_rows, t0 + u.run);
      int32_t cur = 0;
      uint32_t kept = 0u;
      if (u.pos != nullptr) {
        // first index a with pos[a] >= t0 (num_pos if none), kept within [lo, hi]; with
        // a sorted map the probes below t0 form a prefix of the lanes
        int32_t lo = 0, hi = u.num_pos;
        while (hi - lo >= 32) {
          const int32_t step = (hi - lo + 31) / 32;
          const int32_t idx = lo + lane * step;
          const bool below = idx < hi && LDX(u.pos + idx) < t0;
          const int n = __popc(__ballot_sync(0xFFFFFFFFu, below));
          if (n == 0) {
            hi = lo;
          } else {
            hi = min(hi, lo + n * step);
            lo = lo + (n - 1) * step + 1;
          }
        }
        const bool below = lo + lane < hi && LDX(u.pos + lo + lane) < t0;
        cur = lo + __popc(__ballot_sync(0xFFFFFFFFu, below));
        const int32_t pv = cur + lane < u.num_pos ? LDX(u.pos + cur + lane) : t1;
        kept = __reduce_or_sync(0xFFFFFFFFu, (pv >= t0 && pv < t1) ? (1u << (pv - t0)) : 0u);
      }
      if (!active) continue;
      const uint32_t rend = static_cast<uint32_t>(t1) * u.H;
      // two rows a step: both rows' payload and prev loads are issued before either
      // row is combined and stored
      for (uint32_t row = static_cast<uint32_t>(t0) * u.H + sub; row < rend; row += 2 * kRowsPerWarp) {
        uint32_t t[2], h[2];
        int64_t p[2];
        bool ok[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t rk = row + k * kRowsPerWarp;
          ok[k] = rk < rend;
          u.div_h.divmod(ok[k] ? rk : row, t[k], h[k]);
          p[k] = t[k];
          if (u.pos != nullptr) {
            const uint32_t bit = t[k] - static_cast<uint32_t>(t0);
            // both arms signed: -1 must stay negative
            p[k] = ((kept >> bit) & 1u) ? static_cast<int64_t>(cur + __popc(kept & ((1u << bit) - 1u)))
                                        : static_cast<int64_t>(-1);
          }
        }
        uint32_t w[2][BPL][8], q[2][BPL][8];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (!ok[k]) continue;
          if (p[k] >= 0) decode_blocks<kFmt, BPL>(u, p[k], static_cast<int32_t>(h[k]), b0, w[k]);
          const uint16_t* pv =
              u.prev + static_cast<int64_t>(t[k]) * u.prev_row_pitch + static_cast<int64_t>(h[k]) * u.prev_head_pitch;
#pragma unroll
          for (int j = 0; j < BPL; ++j) load32B<kV8, true>(pv + 16 * (b0 + j), q[k][j]);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (!ok[k]) continue;
          uint16_t* out = u.y + static_cast<int64_t>(t[k]) * u.y_row_pitch + static_cast<int64_t>(h[k]) * u.y_head_pitch;
#pragma unroll
          for (int j = 0; j < BPL; ++j) {
            if (p[k] >= 0) {
#pragma unroll
              for (int i = 0; i < 8; ++i) q[k][j][i] = bf16x2_add(q[k][j][i], w[k][j][i]);
            }
            store32B<kV8>(out + 16 * (b0 + j), q[k][j]);
          }
        }
      }
    }
    return;
  }
  if (b0 >= u.nb) return;  // no shuffles below: idle lanes may leave

  const uint32_t stride = nwarps * kRowsPerWarp;
  for (uint32_t row = gwarp * kRowsPerWarp + sub; row < u.total_rows; row += stride) {
    uint32_t r, h;
    u.div_h.divmod(row, r, h);
    uint32_t w[BPL][8];
    if constexpr (kMode == 0) {  // unpack
      decode_blocks<kFmt, BPL>(u, r, static_cast<int32_t>(h), b0, w);
      uint16_t* y = u.y + static_cast<int64_t>(r) * u.y_row_pitch + static_cast<int64_t>(h) * u.y_head_pitch;
#pragma unroll
      for (int j = 0; j < BPL; ++j) store32B<kV8>(y + 16 * (b0 + j), w[j]);
    } else {  // residual in place: row r is the compact index p
      int64_t t = r;
      if (u.pos != nullptr) {
        t = LDX(u.pos + r);
        if (h == 0 && li == 0 && r > 0 && LDX(u.pos + r - 1) >= t) set_status(u.status, 4u);
        if (t < 0 || t >= u.src_rows) {
          if (h == 0 && li == 0) set_status(u.status, 4u);
          continue;
        }
      }
      decode_blocks<kFmt, BPL>(u, r, static_cast<int32_t>(h), b0, w);
      add_store<kV8, false, BPL>(u.prev + t * u.prev_row_pitch + static_cast<int64_t>(h) * u.prev_head_pitch,
                                 u.y + t * u.y_row_pitch + static_cast<int64_t>(h) * u.y_head_pitch, b0, w,
                                 true);
    }
  }
}

// INT4 K payloads, unpack: a column task is (group of G rows, head, 8-channel chunk);
// its FP16 minimum and scale are read once.  RS = G / RPL lanes share a task; each
// loads the codes of its RPL rows together (4 bytes per row), then writes 16 bytes of
// bf16 per row.  A warp holds 32/RS consecutive chunks of a row, so every row access is
// one coalesced span.  (The residual decodes of INT4 K run the row-wise payload kernel.)
template <int RS, int RPL>
__global__ void __launch_bounds__(kThreads) int4_key_decode_kernel(const UnpackParams u) {
  constexpr int CW = 32 / RS;
  const int lane = threadIdx.x & 31;
  const int rs = lane / CW;
  const int cl = lane % CW;
  const PayloadRef& P = u.pay;
  const int32_t nchunk = u.D / 8;
  const int32_t ngroups = (P.rows + P.G - 1) / P.G;
  const int64_t ntask = static_cast<int64_t>(ngroups) * u.H * nchunk;
  const int64_t nwtask = (ntask + CW - 1) / CW;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  // task -> (group, head, chunk): multiply-shift divisions while the task count is
  // below 2^31 (always, short of tensors near the memory size), else 64-bit ones
  const bool small = ntask < (int64_t{1} << 31);
  const FastDiv div_c(static_cast<uint32_t>(nchunk));  // built once per thread
  for (int64_t wt = blockIdx.x * static_cast<int64_t>(kThreads / 32) + threadIdx.x / 32; wt < nwtask;
       wt += nwarps) {
    const int64_t task = wt * CW + cl;
    if (task >= ntask) continue;  // no shuffles in this kernel
    int32_t chunk, h, g;
    if (small) {
      uint32_t gh, c, gg, hh;
      div_c.divmod(static_cast<uint32_t>(task), gh, c);
      u.div_h.divmod(gh, gg, hh);
      chunk = static_cast<int32_t>(c);
      h = static_cast<int32_t>(hh);
      g = static_cast<int32_t>(gg);
    } else {
      chunk = static_cast<int32_t>(task % nchunk);
      h = static_cast<int32_t>((task / nchunk) % u.H);
      g = static_cast<int32_t>(task / (static_cast<int64_t>(nchunk) * u.H));
    }
    const int32_t r0 = g * P.G;
    const int32_t r1 = min(P.rows, r0 + P.G);
    const int32_t col = chunk * 8;
    const int64_t m = (static_cast<int64_t>(g) * u.H + h) * u.D + col;
    uint32_t a[4], c[4];
    load16B(static_cast<const uint16_t*>(P.meta0) + m, a);
    load16B(static_cast<const uint16_t*>(P.meta1) + m, c);
    // all code loads of this lane's rows first
    uint32_t cw[RPL];
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int32_t r = r0 + rs + k * RS;
      if (r < r1) cw[k] = LDX(reinterpret_cast<const uint32_t*>(P.codes + (static_cast<int64_t>(r) * u.H + h) * (u.D / 2) + col / 2));
    }
    float mn[8], sc[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mn[2 * i] = f16_bits_to_f32(static_cast<uint16_t>(a[i] & 0xFFFFu));
      mn[2 * i + 1] = f16_bits_to_f32(static_cast<uint16_t>(a[i] >> 16));
      sc[2 * i] = f16_bits_to_f32(static_cast<uint16_t>(c[i] & 0xFFFFu));
      sc[2 * i + 1] = f16_bits_to_f32(static_cast<uint16_t>(c[i] >> 16));
    }
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int32_t r = r0 + rs + k * RS;
      if (r >= r1) continue;
      uint32_t y[4];
      int4_decode8(cw[k], mn, sc, y);
      store16B(u.y + static_cast<int64_t>(r) * u.y_row_pitch + static_cast<int64_t>(h) * u.y_head_pitch + col, y);
    }
  }
}

template <int RS, int RPL>
cudaError_t key_decode_launch(const UnpackParams& u, int64_t ntask, cudaStream_t s) {
  auto k = int4_key_decode_kernel<RS, RPL>;
  const int occ = cached_occupancy(reinterpret_cast<const void*>(k), kThreads, 0);
  const int64_t warps = (ntask + 32 / RS - 1) / (32 / RS);
  int64_t need = (warps + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = static_cast<int64_t>(num_sms()) * occ * 2;
  if (need < 1) need = 1;
  const int grid = static_cast<int>(need < cap ? need : cap);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("int4_key_decode_kernel", s, k<<<grid, kThreads, 0, s>>>(u); e = cudaGetLastError());
  return e;
}

cudaError_t key_decode_dispatch(const UnpackParams& u, cudaStream_t s) {
  const int64_t ntask = static_cast<int64_t>((u.pay.rows + u.pay.G - 1) / u.pay.G) * u.H * (u.D / 8);
  switch (u.pay.G) {  // RS = G / RPL lanes per column task
    case 16: return key_decode_launch<2, 8>(u, ntask, s);
    case 32: return key_decode_launch<4, 8>(u, ntask, s);
    case 64: return key_decode_launch<8, 8>(u, ntask, s);
    case 128: return key_decode_launch<16, 8>(u, ntask, s);
    case 256: return key_decode_launch<32, 8>(u, ntask, s);
    case 512: return key_decode_launch<32, 16>(u, ntask, s);
  }
  return cudaErrorInvalidValue;
}

template <int L, int BPL, bool kV8, int kFmt, int kMode>
cudaError_t pl_launch(const UnpackParams& u, cudaStream_t s) {
  auto k = payload_kernel<L, BPL, kV8, kFmt, kMode>;
  const int occ = cached_occupancy(reinterpret_cast<const void*>(k), kThreads, 0);
  int64_t need;
  if (kMode == 2)  // one warp per run of u.run tokens
    need = ((static_cast<int64_t>(u.src_rows) + u.run - 1) / u.run + kThreads / 32 - 1) / (kThreads / 32);
  else
    need = (static_cast<int64_t>(u.total_rows) + (kThreads / 32) * (32 / L) - 1) / ((kThreads / 32) * (32 / L));
  const int64_t cap = static_cast<int64_t>(num_sms()) * occ * 2;
  if (need < 1) need = 1;
  const int grid = static_cast<int>(need < cap ? need : cap);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("payload_kernel", s, k<<<grid, kThreads, 0, s>>>(u); e = cudaGetLastError());
  return e;
}

template <int L, int BPL, bool kV8, int kFmt>
cudaError_t pl_dispatch_mode(const UnpackParams& u, cudaStream_t s) {
  switch (u.mode) {
    case 0: return pl_launch<L, BPL, kV8, kFmt, 0>(u, s);
    case 1: return pl_launch<L, BPL, kV8, kFmt, 1>(u, s);
    case 2: return pl_launch<L, BPL, kV8, kFmt, 2>(u, s);
  }
  return cudaErrorInvalidValue;
}

template <int L, int BPL, bool kV8>
cudaError_t pl_dispatch_fm(const UnpackParams& u, cudaStream_t s) {
  switch (u.pay.fmt) {
    case 1: return pl_dispatch_mode<L, BPL, kV8, 1>(u, s);
    case 2: return pl_dispatch_mode<L, BPL, kV8, 2>(u, s);
    case 3: return pl_dispatch_mode<L, BPL, kV8, 3>(u, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_payload_decode(const UnpackParams& u_in, int /*lanes*/, bool v8, cudaStream_t s) {
  UnpackParams u = u_in;
  // copy mode: runs of 4..32 tokens, about 32 runs per SM
  const int64_t per = (static_cast<int64_t>(u.src_rows) + num_sms() * 32 - 1) / (num_sms() * 32);
  u.run = static_cast<int32_t>(per < 4 ? 4 : (per > 32 ? 32 : per));
  // INT4 K unpack runs column-wise; the residual decodes run row by row like every other
  // payload (in place, the row-wise kernel measured 3% faster than a column-wise one)
  if (u.pay.fmt == 2 && u.pay.kind == 0 && u.mode == 0) return key_decode_dispatch(u, s);
  const int bpl = (u.nb % 2 == 0) ? 2 : 1;
  int lanes = 1;
  while (lanes < u.nb / bpl) lanes <<= 1;
#define KVQ_PL(LN, B)                                                                          \
  if (lanes == LN && bpl == B)                                                                 \
    return v8 ? pl_dispatch_fm<LN, B, true>(u, s) : pl_dispatch_fm<LN, B, false>(u, s);
  KVQ_PL(1, 1) KVQ_PL(2, 1) KVQ_PL(4, 1) KVQ_PL(8, 1) KVQ_PL(16, 1) KVQ_PL(32, 1)
  KVQ_PL(1, 2) KVQ_PL(2, 2) KVQ_PL(4, 2) KVQ_PL(8, 2) KVQ_PL(16, 2)
#undef KVQ_PL
  return cudaErrorInvalidValue;
}

}  // namespace kvq
