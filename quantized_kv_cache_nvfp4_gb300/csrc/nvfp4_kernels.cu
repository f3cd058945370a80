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
// Dividing by s itself when 1 / s is infinite is the tiny-scale rule of "vllm-rlt
// PR #166: INT4 KV packing ...", Purpose.
//
// FP8 E4M3 rows ("feat(kvcache): ... (FreeToken PR #408)", fp8 store notes) take the
// same kernels with kFmt = 3: rs = amax / 448; q = x * (1 / rs) (x / rs when the
// reciprocal overflows); code = e4m3(q) nearest even; decode y = bf16(e4m3 * rs);
// D code bytes per row and no block scales.
//
// Work mapping: a lane owns BPL consecutive 16-element blocks of a row (BPL = 2 when
// the row has an even number of blocks: two 256-bit loads, 64 contiguous bytes per
// lane).  The L lanes of a row (L = next power of two of D/16/BPL) form an aligned
// sub-warp, so the row amax is a log2(L)-step xor butterfly.  A warp handles 32/L
// rows per iteration (at D256, H4: exactly the four heads of one token); a grid-stride
// loop issues the next row's loads before the current row's arithmetic.  No tensor
// cores: nothing here is a contraction.
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

// The BPL source blocks of this lane for one row (zeros past the row's end).
// Residual mode builds bf16(cur - prev) for the row at position pos[p].
template <int kMode, bool kV8, int BPL>
__device__ __forceinline__ void load_source(const EncodeParams& p, const RowLoc& loc, int b0,
                                            uint32_t (&w)[BPL][8]) {
  const EncodeTensor& T = p.ten[loc.tensor];
  int64_t src = loc.tok;
  if constexpr (kMode == kEncResidual) {
    if (p.pos != nullptr) src = LDX(p.pos + loc.tok);
    if (src < 0 || src >= p.src_rows) {  // a zero residual row
#pragma unroll
      for (int j = 0; j < BPL; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) w[j][i] = 0u;
      return;
    }
  }
  const uint16_t* x = T.x + src * T.row_pitch + static_cast<int64_t>(loc.h) * T.head_pitch;
#pragma unroll
  for (int j = 0; j < BPL; ++j) {
    if (b0 + j < p.nb) {
      load32B<kV8, true>(x + 16 * (b0 + j), w[j]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = 0u;
    }
  }
  if constexpr (kMode == kEncResidual) {
    const uint16_t* q = T.prev + src * T.prev_row_pitch + static_cast<int64_t>(loc.h) * T.prev_head_pitch;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      if (b0 + j >= p.nb) continue;
      uint32_t pw[8];
      load32B<kV8, true>(q + 16 * (b0 + j), pw);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[j][i] = bf16x2_sub(w[j][i], pw[i]);
    }
  }
}


template <int L, int BPL, bool kV8, int kMode, int kMinBlocks, int kFmt>
__global__ void __launch_bounds__(kThreads, kMinBlocks) nvfp4_encode_kernel(const EncodeParams p) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int li = lane % L;
  const int sub = lane / L;
  const int b0 = li * BPL;
  const uint32_t total = p.rows_per_tensor * static_cast<uint32_t>(p.ntensors);
  const uint32_t nwarps = gridDim.x * (kThreads / 32);
  const uint32_t stride = nwarps * kRowsPerWarp;
  uint32_t row = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
  const bool lane_active = b0 < p.nb;

  uint32_t w[BPL][8];
#pragma unroll
  for (int j = 0; j < BPL; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) w[j][i] = 0u;
  if (lane_active && row < total)
    load_source<kMode, kV8, BPL>(p, locate(row, p.rows_per_tensor, p.div_h), b0, w);

  // The loop bound is uniform across the warp (row - sub is), so every lane runs
  // every shuffle of every iteration.
  for (; row - sub < total; row += stride) {
    const bool valid = row < total;
    const RowLoc loc = locate(valid ? row : 0u, p.rows_per_tensor, p.div_h);

    // issue the next row's loads before this row's arithmetic
    uint32_t nw[BPL][8];
#pragma unroll
    for (int j = 0; j < BPL; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) nw[j][i] = 0u;
    const uint32_t nrow = row + stride;
    if (lane_active && nrow < total)
      load_source<kMode, kV8, BPL>(p, locate(nrow, p.rows_per_tensor, p.div_h), b0, nw);

    // destination row and skip decision
    int64_t drow = static_cast<int64_t>(loc.tok) * p.H + loc.h;
    bool skip = !valid;
    if constexpr (kMode == kEncScatter) {
      if (valid) {
        const int64_t slot = LDX(p.slot_ids + loc.tok);
        if (slot < 0) {
          skip = true;
        } else if (slot >= p.num_slots) {
          skip = true;
          if (loc.h == 0 && li == 0 && loc.tensor == 0) set_status(p.status, 1u);
        } else {
          drow = slot * p.H + loc.h;
        }
      }
    }
    if constexpr (kMode == kEncResidual) {
      if (valid && loc.h == 0 && li == 0 && loc.tensor == 0 && p.pos != nullptr) {
        const int32_t ps = LDX(p.pos + loc.tok);
        bool bad = ps < 0 || ps >= p.src_rows;
        if (loc.tok > 0 && LDX(p.pos + loc.tok - 1) >= ps) bad = true;
        if (bad) set_status(p.status, 4u);
        if (p.pos_out != nullptr) STX(p.pos_out + loc.tok, ps);
      }
    }

    // row scale
    float vb[BPL];
    float lmax = 0.0f;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      vb[j] = absmax16(w[j]);  // zero for blocks past the row's end
      lmax = fmaxf(lmax, vb[j]);
    }
    const float amax = group_max<L>(lmax);
    if constexpr (kFmt == 3) {  // FP8 E4M3: one scale per row, no block scales
      const float rs = __fdiv_rn(amax, kE4M3Max);
      const float inv = (rs != 0.0f) ? __frcp_rn(rs) : 0.0f;
      uint32_t c8[BPL][4];
#pragma unroll
      for (int j = 0; j < BPL; ++j) fp8_quantize16(w[j], rs, inv, c8[j]);
      if (!skip && lane_active) {
        const Nvfp4Planes& d = p.ten[loc.tensor].dst;
        uint8_t* cp = d.codes + drow * (16 * p.nb) + 16 * b0;
#pragma unroll
        for (int j = 0; j < BPL; ++j) store16B(cp + 16 * j, c8[j]);
        if (li == 0) STX(d.rscale + drow, rs);
      }
#pragma unroll
      for (int j = 0; j < BPL; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) w[j][i] = nw[j][i];
      continue;
    }
    const float rs = __fdiv_rn(amax, kE2M1Max * kE4M3Max);
    const float rinv = (rs != 0.0f) ? __frcp_rn(rs) : 0.0f;

    uint32_t c[BPL][2];
    uint32_t bsb[BPL];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      bsb[j] = block_scale_code(vb[j], rs, rinv);
      const float s = __fmul_rn(e4m3_to_f32(bsb[j]), rs);
      quantize_block(w[j], s, c[j][0], c[j][1]);
    }

    if (!skip && lane_active) {
      const Nvfp4Planes& d = p.ten[loc.tensor].dst;
      uint8_t* cp = d.codes + drow * (8 * p.nb) + 8 * b0;
      uint8_t* bp = d.bscale + drow * p.nb + b0;
      if constexpr (BPL == 2) {
        const uint32_t cw[4] = {c[0][0], c[0][1], c[1][0], c[1][1]};
        store16B(cp, cw);
        STX(reinterpret_cast<uint16_t*>(bp), static_cast<uint16_t>(bsb[0] | (bsb[1] << 8)));
      } else {
        store8B(cp, c[0][0], c[0][1]);
        STX(bp, static_cast<uint8_t>(bsb[0]));
      }
      if (li == 0) STX(d.rscale + drow, rs);
    }

#pragma unroll
    for (int j = 0; j < BPL; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = nw[j][i];
  }
}

// Restore one row (or skip it): resolve the slot through the block table.
struct RestoreRow {
  int64_t srow;  // pool row (slot * H + h), or -1 to skip
  uint16_t* y;   // first element of the output row
  const DecodeTensor* ten;
};

template <int kMode>
__device__ __forceinline__ RestoreRow resolve_row(const DecodeParams& p, uint32_t row, int li) {
  RestoreRow r{-1, nullptr, nullptr};
  const int tensor = row >= p.rows_per_tensor ? 1 : 0;
  const uint32_t rr = row - (tensor ? p.rows_per_tensor : 0u);
  uint32_t orow, h;
  p.div_h.divmod(rr, orow, h);
  const DecodeTensor& T = p.ten[tensor];
  if constexpr (kMode == kDecRestore) {
    uint32_t s, t;
    p.div_tmax.divmod(orow, s, t);
    const int32_t len = LDX(p.seq_lens + s);
    if (len < 0 || len > p.seq_cap) {
      if (t == 0 && h == 0 && li == 0 && tensor == 0) set_status(p.status, 8u);
      return r;
    }
    if (static_cast<int32_t>(t) >= len) return r;
    uint32_t blk_i, off;
    p.div_bs.divmod(t, blk_i, off);
    const int32_t blk = LDX(p.block_table + static_cast<int64_t>(s) * p.max_blocks + blk_i);
    if (blk < 0 || blk >= p.num_blocks) {
      if (h == 0 && li == 0 && tensor == 0) set_status(p.status, 2u);
      return r;
    }
    r.srow = (static_cast<int64_t>(blk) * p.block_size + off) * p.H + h;
  } else {
    r.srow = rr;
  }
  r.y = T.y + static_cast<int64_t>(orow) * T.row_pitch + static_cast<int64_t>(h) * T.head_pitch;
  r.ten = &T;
  return r;
}

// The restore's index loads of one row, issued ahead of the row: its sequence length
// and block-table entry (both addressed from the row number alone), checked later.
struct RowFetch {
  uint32_t row;
  int32_t len, blk;
};

__device__ __forceinline__ int32_t ld_i32_ahead(const int32_t* p) {
  if (!KVQ_OK(p, 4, 4)) return -1;
  int32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ RowFetch fetch_row(const DecodeParams& p, uint32_t row, uint32_t total) {
  RowFetch f{row, -1, -1};
  if (row >= total) return f;
  const int tensor = row >= p.rows_per_tensor ? 1 : 0;
  const uint32_t rr = row - (tensor ? p.rows_per_tensor : 0u);
  uint32_t orow, h, s, t, bi, off;
  p.div_h.divmod(rr, orow, h);
  p.div_tmax.divmod(orow, s, t);
  p.div_bs.divmod(t, bi, off);
  f.len = ld_i32_ahead(p.seq_lens + s);
  if (bi < static_cast<uint32_t>(p.max_blocks)) f.blk = ld_i32_ahead(p.block_table + static_cast<int64_t>(s) * p.max_blocks + bi);
  return f;
}

__device__ __forceinline__ RestoreRow finish_row(const DecodeParams& p, const RowFetch& f, int li) {
  RestoreRow r{-1, nullptr, nullptr};
  const int tensor = f.row >= p.rows_per_tensor ? 1 : 0;
  const uint32_t rr = f.row - (tensor ? p.rows_per_tensor : 0u);
  uint32_t orow, h, s, t, bi, off;
  p.div_h.divmod(rr, orow, h);
  p.div_tmax.divmod(orow, s, t);
  if (f.len < 0 || f.len > p.seq_cap) {
    if (t == 0 && h == 0 && li == 0 && tensor == 0) set_status(p.status, 8u);
    return r;
  }
  if (static_cast<int32_t>(t) >= f.len) return r;
  p.div_bs.divmod(t, bi, off);
  if (f.blk < 0 || f.blk >= p.num_blocks) {
    if (h == 0 && li == 0 && tensor == 0) set_status(p.status, 2u);
    return r;
  }
  const DecodeTensor& T = p.ten[tensor];
  r.srow = (static_cast<int64_t>(f.blk) * p.block_size + off) * p.H + h;
  r.y = T.y + static_cast<int64_t>(orow) * T.row_pitch + static_cast<int64_t>(h) * T.head_pitch;
  r.ten = &T;
  return r;
}

// R rows per lane per iteration: all R block-table lookups, then all R code loads,
// then the arithmetic and stores, so R dependent load chains are in flight at once.
template <int L, int BPL, bool kV8, int kMode, int R, int kMinBlocks, int kFmt>
__global__ void __launch_bounds__(kThreads, kMinBlocks) nvfp4_decode_kernel(const DecodeParams p) {
  constexpr int kRowsPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int li = lane % L;
  const int sub = lane / L;
  const int b0 = li * BPL;
  const uint32_t total = p.rows_per_tensor * static_cast<uint32_t>(p.ntensors);
  const uint32_t stride = gridDim.x * (kThreads / 32) * kRowsPerWarp;
  if (b0 >= p.nb) return;  // no shuffles below: idle lanes may leave

  const uint32_t first = (blockIdx.x * (kThreads / 32) + threadIdx.x / 32) * kRowsPerWarp + sub;
  // FP8 restore: the next iteration's index loads are issued an iteration ahead (its
  // rows are short, so the index chain is a large part of each row's latency; for
  // NVFP4 it measured neither faster nor slower and the rows resolve in place)
  constexpr bool kAhead = kMode == kDecRestore && kFmt == 3;
  RowFetch fn[R];
  if constexpr (kAhead) {
#pragma unroll
    for (int r = 0; r < R; ++r) fn[r] = fetch_row(p, first + r * stride, total);
  }
  for (uint32_t row0 = first; row0 < total; row0 += R * stride) {
    RestoreRow rr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t row = row0 + r * stride;
      if constexpr (kAhead) {
        rr[r] = (row < total) ? finish_row(p, fn[r], li) : RestoreRow{-1, nullptr, nullptr};
      } else {
        rr[r] = (row < total) ? resolve_row<kMode>(p, row, li) : RestoreRow{-1, nullptr, nullptr};
      }
    }
    if constexpr (kAhead) {
#pragma unroll
      for (int r = 0; r < R; ++r) fn[r] = fetch_row(p, row0 + (R + r) * stride, total);
    }
    if constexpr (kFmt == 3) {  // FP8 E4M3 rows: 16 code bytes per block, one scale
      uint32_t c8[R][BPL][4];
      float rs8[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (rr[r].srow < 0) continue;
        const DecodeTensor& T = *rr[r].ten;
        rs8[r] = LDX(T.rscale + rr[r].srow);
#pragma unroll
        for (int j = 0; j < BPL; ++j) load16B(T.codes + rr[r].srow * (16 * p.nb) + 16 * (b0 + j), c8[r][j]);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (rr[r].srow < 0) continue;
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
          fp8_decode16(c8[r][j], rs8[r], out);
          store32B<kV8>(rr[r].y + 16 * (b0 + j), out);
        }
      }
    } else {
      uint32_t cw[R][2 * BPL];
      uint32_t bsb[R];
      float rs[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (rr[r].srow < 0) continue;
        const DecodeTensor& T = *rr[r].ten;
        const int64_t srow = rr[r].srow;
        rs[r] = LDX(T.rscale + srow);
        if constexpr (BPL == 2) {
          uint32_t c4[4];
          load16B(T.codes + srow * (8 * p.nb) + 8 * b0, c4);
#pragma unroll
          for (int i = 0; i < 4; ++i) cw[r][i] = c4[i];
          bsb[r] = LDX(reinterpret_cast<const uint16_t*>(T.bscale + srow * p.nb + b0));
        } else {
          load8B(T.codes + srow * (8 * p.nb) + 8 * b0, cw[r][0], cw[r][1]);
          bsb[r] = LDX(T.bscale + srow * p.nb + b0);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (rr[r].srow < 0) continue;
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
          nvfp4_decode16(cw[r][2 * j], cw[r][2 * j + 1], (bsb[r] >> (8 * j)) & 0xFFu, rs[r], out);
          store32B<kV8>(rr[r].y + 16 * (b0 + j), out);
        }
      }
    }
  }
}

// Grid of a grid-stride kernel: enough blocks for every row, at most `factor`
// times the number of blocks that can be resident at once (SMs x occupancy).
template <typename K>
int grid_for(K kernel, uint32_t rows, int rows_per_cta, int factor) {
  const int occ = cached_occupancy(reinterpret_cast<const void*>(kernel), kThreads, 0);
  int64_t need = (static_cast<int64_t>(rows) + rows_per_cta - 1) / rows_per_cta;
  int64_t cap = static_cast<int64_t>(num_sms()) * occ * factor;
  if (need < 1) need = 1;
  return static_cast<int>(need < cap ? need : cap);
}

// Launch shapes (measured on the 1M-token workload; see the profiles): the encode
// targets 4 resident blocks per SM; the restore handles two rows per lane per
// iteration and launches twice as many blocks as can be resident at once.
constexpr int kEncMinBlocks = 4;
constexpr int kEncGridFactor = 2;
constexpr int kDecRows = 2;
constexpr int kDecMinBlocks = 1;
constexpr int kDecGridFactor = 2;

template <int L, int BPL, bool kV8, int kMode, int kFmt>
cudaError_t enc_launch(const EncodeParams& p, cudaStream_t s) {
  auto k = nvfp4_encode_kernel<L, BPL, kV8, kMode, kEncMinBlocks, kFmt>;
  uint32_t rows = p.rows_per_tensor * p.ntensors;
  int grid = grid_for(k, rows, (kThreads / 32) * (32 / L), kEncGridFactor);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("nvfp4_encode_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

template <int L, int BPL, bool kV8, int kMode, int kFmt>
cudaError_t dec_launch(const DecodeParams& p, cudaStream_t s) {
  auto k = nvfp4_decode_kernel<L, BPL, kV8, kMode, kDecRows, kDecMinBlocks, kFmt>;
  uint32_t rows = p.rows_per_tensor * p.ntensors;
  int grid = grid_for(k, rows, (kThreads / 32) * (32 / L) * kDecRows, kDecGridFactor);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("nvfp4_decode_kernel", s, k<<<grid, kThreads, 0, s>>>(p); e = cudaGetLastError());
  return e;
}

// Lanes per row and blocks per lane for nb = D / 16 blocks.
void row_shape(int nb, int& lanes, int& bpl) {
  bpl = (nb % 2 == 0) ? 2 : 1;
  const int per = nb / bpl;
  lanes = 1;
  while (lanes < per) lanes <<= 1;
}

#define KVQ_SHAPES(X) X(1, 1) X(2, 1) X(4, 1) X(8, 1) X(16, 1) X(32, 1) \
                      X(1, 2) X(2, 2) X(4, 2) X(8, 2) X(16, 2)

template <int kMode, int kFmt>
cudaError_t enc_dispatch(const EncodeParams& p, bool v8, cudaStream_t s) {
  int lanes, bpl;
  row_shape(p.nb, lanes, bpl);
#define KVQ_ENC(LN, B)                                                                    \
  if (lanes == LN && bpl == B)                                                            \
    return v8 ? enc_launch<LN, B, true, kMode, kFmt>(p, s) : enc_launch<LN, B, false, kMode, kFmt>(p, s);
  KVQ_SHAPES(KVQ_ENC)
#undef KVQ_ENC
  return cudaErrorInvalidValue;
}

template <int kMode, int kFmt>
cudaError_t dec_dispatch(const DecodeParams& p, bool v8, cudaStream_t s) {
  int lanes, bpl;
  row_shape(p.nb, lanes, bpl);
#define KVQ_DEC(LN, B)                                                                    \
  if (lanes == LN && bpl == B)                                                            \
    return v8 ? dec_launch<LN, B, true, kMode, kFmt>(p, s) : dec_launch<LN, B, false, kMode, kFmt>(p, s);
  KVQ_SHAPES(KVQ_DEC)
#undef KVQ_DEC
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_nvfp4_encode(const EncodeParams& p, int mode, int fmt, bool v8, cudaStream_t s) {
  const bool fp8 = fmt == 3;
  switch (mode) {
    case kEncScatter:
      return fp8 ? enc_dispatch<kEncScatter, 3>(p, v8, s) : enc_dispatch<kEncScatter, 1>(p, v8, s);
    case kEncPack:
      return fp8 ? enc_dispatch<kEncPack, 3>(p, v8, s) : enc_dispatch<kEncPack, 1>(p, v8, s);
    case kEncResidual:
      return fp8 ? enc_dispatch<kEncResidual, 3>(p, v8, s) : enc_dispatch<kEncResidual, 1>(p, v8, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_nvfp4_decode(const DecodeParams& p, int mode, int fmt, bool v8, cudaStream_t s) {
  if (mode != kDecRestore) return cudaErrorInvalidValue;
  return fmt == 3 ? dec_dispatch<kDecRestore, 3>(p, v8, s) : dec_dispatch<kDecRestore, 1>(p, v8, s);
}

}  // namespace kvq
