// nvfp4_kernels.cu -- NVFP4 row codec kernels for sm_103a.
//
// Format ("feat(kvcache): add nvfp4 kv quantization (FreeToken PR #408)", Summary
// and codec-delta port note): each (token, KV head) row of D bf16 becomes D/2 bytes
// of E2M1 nibbles (low nibble = even element), D/16 E4M3 block scales and one FP32
// row scale; elements are quantised against the STORED (rounded) block scale.
//
// Arithmetic, per row, in this order (all binary32, nearest even):
//   amax = max |x|;  rs = amax / 2688                      (2688 = 6 * 448)
//   per 16-block: vb = max |x|;  t = min((vb / 6) / rs, 448)  (t = 0 when rs == 0)
//                 bs = e4m3(t) (nearest even);  s = bs * rs
//                 inv = 1 / s (0 when s == 0);  q = x * inv, or x / s when inv is inf
//                 code = e2m1(q) (nearest even, saturating at 6, sign of x)
//   decode: y = bf16((e2m1 * bs) * rs)  (the inner product is exact)
// The tiny-scale direct division follows "vllm-rlt PR #166: INT4 KV packing ...",
// Purpose ("a direct-division fallback when their reciprocal overflows").
//
// Work mapping: one lane owns one 16-element block (32 bytes of bf16, one 256-bit
// load when aligned); the D/16 lanes of a row form an aligned sub-warp of L lanes
// (L = next power of two), so the row amax is a log2(L)-step xor butterfly.  A
// warp therefore handles 32/L rows per iteration; a grid-stride loop with the next
// row's load issued before the current row's arithmetic keeps two loads in flight
// per lane.  No tensor cores: nothing here is a contraction.
#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;

struct RowLoc {
  int tensor;     // 0 = K, 1 = V
  uint32_t tok;   // token (or compact row)
  uint32_t h;
};

__device__ __forceinline__ RowLoc locate(uint32_t row, uint32_t rows_per_tensor, const FastDiv& dh) {
  RowLoc r;
  r.tensor = row >= rows_per_tensor ? 1 : 0;
  uint32_t rr = row - (r.tensor ? rows_per_tensor : 0u);
  dh.divmod(rr, r.tok, r.h);
  return r;
}

// Source block of 16 bf16 for (row, block b).  Residual mode builds
// bf16(cur - prev) for the row at position pos[p].
template <int kMode, bool kV8>
__device__ __forceinline__ bool load_source(const EncodeParams& p, const RowLoc& loc, int b,
                                            uint32_t (&w)[8]) {
  const EncodeTensor& T = p.ten[loc.tensor];
  if constexpr (kMode == kEncResidual) {
    int64_t src = loc.tok;
    if (p.pos != nullptr) src = LDX(p.pos + loc.tok);
    if (src < 0 || src >= p.src_rows) {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = 0u;  // a zero residual row
      return false;
    }
    uint32_t c[8], q[8];
    load32B<kV8, true>(T.x + src * T.row_pitch + loc.h * T.head_pitch + 16 * b, c);
    load32B<kV8, true>(T.prev + src * T.prev_row_pitch + loc.h * T.prev_head_pitch + 16 * b, q);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float lo = __fsub_rn(bf16lo(c[i]), bf16lo(q[i]));
      float hi = __fsub_rn(bf16hi(c[i]), bf16hi(q[i]));
      w[i] = pack_bf16x2(lo, hi);
    }
    return true;
  } else {
    load32B<kV8, true>(T.x + static_cast<int64_t>(loc.tok) * T.row_pitch +
                           static_cast<int64_t>(loc.h) * T.head_pitch + 16 * b,
                       w);
    return true;
  }
}

template <int L, bool kV8, int kMode>
__global__ void __launch_bounds__(kThreads) nvfp4_encode_kernel(const EncodeParams p) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int b = lane % L;
  const int sub = lane / L;
  const uint32_t total = p.rows_per_tensor * static_cast<uint32_t>(p.ntensors);
  const uint32_t nwarps = gridDim.x * (kThreads / 32);
  const uint32_t stride = nwarps * kRowsPerWarp;
  uint32_t row = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
  const bool lane_has_block = b < p.nb;

  // prefetch the first row
  uint32_t w[8];
  {
    bool act = lane_has_block && row < total;
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0u;
    if (act) load_source<kMode, kV8>(p, locate(row, p.rows_per_tensor, p.div_h), b, w);
  }

  // The loop bound is uniform across the warp (row - sub is), so every lane runs
  // every shuffle of every iteration.
  for (; row - sub < total; row += stride) {
    const bool valid = row < total;
    const RowLoc loc = locate(valid ? row : 0u, p.rows_per_tensor, p.div_h);

    // issue the next row's load before this row's arithmetic
    uint32_t nw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) nw[i] = 0u;
    const uint32_t nrow = row + stride;
    if (lane_has_block && nrow < total)
      load_source<kMode, kV8>(p, locate(nrow, p.rows_per_tensor, p.div_h), b, nw);

    // destination row and skip decision
    int64_t drow = static_cast<int64_t>(loc.tok) * p.H + loc.h;
    bool skip = !valid;
    if constexpr (kMode == kEncScatter) {
      if (valid) {
        int64_t slot = LDX(p.slot_ids + loc.tok);
        if (slot < 0) {
          skip = true;
        } else if (slot >= p.num_slots) {
          skip = true;
          if (loc.h == 0 && b == 0 && loc.tensor == 0) set_status(p.status, 1u);
        } else {
          drow = slot * p.H + loc.h;
        }
      }
    }
    if constexpr (kMode == kEncResidual) {
      if (valid && loc.h == 0 && b == 0 && loc.tensor == 0 && p.pos != nullptr) {
        int32_t ps = LDX(p.pos + loc.tok);
        bool bad = ps < 0 || ps >= p.src_rows;
        if (loc.tok > 0 && LDX(p.pos + loc.tok - 1) >= ps) bad = true;
        if (bad) set_status(p.status, 4u);
        if (p.pos_out != nullptr) STX(p.pos_out + loc.tok, ps);
      }
    }

    // row and block scales
    const float vb = lane_has_block ? absmax16(w) : 0.0f;
    const float amax = group_max<L>(vb);
    const float rs = __fdiv_rn(amax, kE2M1Max * kE4M3Max);
    float t = 0.0f;
    if (rs != 0.0f) t = __fdiv_rn(__fdiv_rn(vb, kE2M1Max), rs);
    t = fminf(t, kE4M3Max);
    const uint32_t bsb = e4m3_from_f32(t);
    const float bs = e4m3_to_f32(bsb);
    const float s = __fmul_rn(bs, rs);
    const float inv = (s != 0.0f) ? __frcp_rn(s) : 0.0f;
    const bool use_div = isinf(inv);

    // element codes, two per byte, low nibble first
    uint32_t c0 = 0u, c1 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xl = bf16lo(w[i]);
      const float xh = bf16hi(w[i]);
      float ql, qh;
      if (use_div) {
        ql = __fdiv_rn(xl, s);
        qh = __fdiv_rn(xh, s);
      } else {
        ql = __fmul_rn(xl, inv);
        qh = __fmul_rn(xh, inv);
      }
      const uint32_t byte = e2m1x2_from_f32(ql, qh);
      if (i < 4)
        c0 |= byte << (8 * i);
      else
        c1 |= byte << (8 * (i - 4));
    }

    if (!skip && lane_has_block) {
      const Nvfp4Planes& d = p.ten[loc.tensor].dst;
      store8B(d.codes + drow * (8 * p.nb) + 8 * b, c0, c1);
      STX(d.bscale + drow * p.nb + b, static_cast<uint8_t>(bsb));
      if (b == 0) STX(d.rscale + drow, rs);
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = nw[i];
  }
}

template <int L, bool kV8, int kMode>
__global__ void __launch_bounds__(kThreads) nvfp4_decode_kernel(const DecodeParams p) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int b = lane % L;
  const int sub = lane / L;
  const uint32_t total = p.rows_per_tensor * static_cast<uint32_t>(p.ntensors);
  const uint32_t stride = gridDim.x * (kThreads / 32) * kRowsPerWarp;
  if (b >= p.nb) return;  // no shuffles below: idle lanes may leave

  for (uint32_t row = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
       row < total; row += stride) {
    const int tensor = row >= p.rows_per_tensor ? 1 : 0;
    const uint32_t rr = row - (tensor ? p.rows_per_tensor : 0u);
    uint32_t orow, h;
    p.div_h.divmod(rr, orow, h);
    int64_t srow;
    if constexpr (kMode == kDecRestore) {
      uint32_t s, t;
      p.div_tmax.divmod(orow, s, t);
      const int32_t len = LDX(p.seq_lens + s);
      if (len < 0 || len > p.seq_cap) {
        if (t == 0 && h == 0 && b == 0 && tensor == 0) set_status(p.status, 8u);
        continue;
      }
      if (static_cast<int32_t>(t) >= len) continue;
      uint32_t blk_i, off;
      p.div_bs.divmod(t, blk_i, off);
      const int32_t blk = LDX(p.block_table + static_cast<int64_t>(s) * p.max_blocks + blk_i);
      if (blk < 0 || blk >= p.num_blocks) {
        if (h == 0 && b == 0 && tensor == 0) set_status(p.status, 2u);
        continue;
      }
      srow = (static_cast<int64_t>(blk) * p.block_size + off) * p.H + h;
    } else {
      srow = rr;
    }
    const DecodeTensor& T = p.ten[tensor];
    uint32_t cw0, cw1;
    load8B(T.codes + srow * (8 * p.nb) + 8 * b, cw0, cw1);
    const uint32_t bsb = LDX(T.bscale + srow * p.nb + b);
    const float rs = LDX(T.rscale + srow);
    const uint32_t bs2 = e4m3_to_f16x2(bsb) & 0xFFFFu;
    const uint32_t bsx2 = bs2 | (bs2 << 16);

    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t byte = ((i < 4 ? cw0 : cw1) >> (8 * (i & 3))) & 0xFFu;
      const uint32_t v2 = hmul2_bits(e2m1x2_to_f16x2(byte), bsx2);  // exact
      float lo, hi;
      f16x2_to_f32(v2, lo, hi);
      out[i] = pack_bf16x2(__fmul_rn(lo, rs), __fmul_rn(hi, rs));
    }
    store32B<kV8>(T.y + static_cast<int64_t>(orow) * T.row_pitch +
                      static_cast<int64_t>(h) * T.head_pitch + 16 * b,
                  out);
  }
}

template <typename K>
int grid_for(K kernel, uint32_t rows, int rows_per_cta) {
  static int per_sm[64] = {0};
  (void)per_sm;
  int occ = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0);
  if (occ < 1) occ = 1;
  int64_t need = (static_cast<int64_t>(rows) + rows_per_cta - 1) / rows_per_cta;
  int64_t cap = static_cast<int64_t>(num_sms()) * occ;
  if (need < 1) need = 1;
  return static_cast<int>(need < cap ? need : cap);
}

template <int L, bool kV8, int kMode>
cudaError_t enc_launch(const EncodeParams& p, cudaStream_t s) {
  auto k = nvfp4_encode_kernel<L, kV8, kMode>;
  uint32_t rows = p.rows_per_tensor * p.ntensors;
  int grid = grid_for(k, rows, (kThreads / 32) * (32 / L));
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("nvfp4_encode_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

template <int L, bool kV8, int kMode>
cudaError_t dec_launch(const DecodeParams& p, cudaStream_t s) {
  auto k = nvfp4_decode_kernel<L, kV8, kMode>;
  uint32_t rows = p.rows_per_tensor * p.ntensors;
  int grid = grid_for(k, rows, (kThreads / 32) * (32 / L));
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("nvfp4_decode_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

template <int kMode>
cudaError_t enc_dispatch(const EncodeParams& p, int lanes, bool v8, cudaStream_t s) {
#define KVQ_ENC(LN)                                                   \
  case LN:                                                            \
    return v8 ? enc_launch<LN, true, kMode>(p, s) : enc_launch<LN, false, kMode>(p, s);
  switch (lanes) {
    KVQ_ENC(1)
    KVQ_ENC(2)
    KVQ_ENC(4)
    KVQ_ENC(8)
    KVQ_ENC(16)
    KVQ_ENC(32)
  }
#undef KVQ_ENC
  return cudaErrorInvalidValue;
}

template <int kMode>
cudaError_t dec_dispatch(const DecodeParams& p, int lanes, bool v8, cudaStream_t s) {
#define KVQ_DEC(LN)                                                   \
  case LN:                                                            \
    return v8 ? dec_launch<LN, true, kMode>(p, s) : dec_launch<LN, false, kMode>(p, s);
  switch (lanes) {
    KVQ_DEC(1)
    KVQ_DEC(2)
    KVQ_DEC(4)
    KVQ_DEC(8)
    KVQ_DEC(16)
    KVQ_DEC(32)
  }
#undef KVQ_DEC
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_nvfp4_encode(const EncodeParams& p, int mode, int lanes, bool v8,
                                cudaStream_t s) {
  switch (mode) {
    case kEncScatter:
      return enc_dispatch<kEncScatter>(p, lanes, v8, s);
    case kEncPack:
      return enc_dispatch<kEncPack>(p, lanes, v8, s);
    case kEncResidual:
      return enc_dispatch<kEncResidual>(p, lanes, v8, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_nvfp4_decode(const DecodeParams& p, int mode, int lanes, bool v8,
                                cudaStream_t s) {
  switch (mode) {
    case kDecRestore:
      return dec_dispatch<kDecRestore>(p, lanes, v8, s);
    case kDecUnpack:
      return dec_dispatch<kDecUnpack>(p, lanes, v8, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
