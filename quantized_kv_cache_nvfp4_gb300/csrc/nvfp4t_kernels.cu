// nvfp4t_kernels.cu -- NVFP4 with one FP32 scale per tensor: the logical layout of
// "vllm-rlt PR #166: INT4 KV packing/unpacking and cross-loop residual reconstruction"
// (Purpose): blocks of 16 values with E4M3 scales plus one FP32 number for the
// whole tensor; K blocks run along 16 token rows at a fixed head and channel, V
// blocks along 16 channels at a fixed token and head; the last block may be short.
//
// rs = amax of the whole tensor / 2688, kept as the decode multiplier; each block of
// 16 takes the row codec's steps against it: block scale e4m3(min((vb/6)/rs, 448)),
// codes e2m1(x * 1/(bs*rs)) (x / (bs*rs) when the reciprocal overflows), decode
// bf16((e2m1 * bs) * rs).
//
// Encoding runs as three kernels on the caller's stream (the scale slot is zeroed by
// a memset first): the tensor's amax, gathered with atomicMax on the float bits into
// the packed tensor's own scale slot (non-negative floats order as their bits); the
// block codes, which read that amax; and one thread that turns the slot into rs.  No
// scratch memory, and safe under graph capture.
#include "kvq_device.cuh"
#include "kvq_params.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;
constexpr float kRowScaleDiv = 2688.0f;  // 6 * 448

// Per-half maximum of magnitudes of two bf16x2 words (the sign bits are cleared by the
// caller); a bf16 maximum is one of its inputs, so nothing rounds.
__device__ __forceinline__ uint32_t absmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void tensor_scale(const float* slot, float& rs, float& rinv) {
  const float amax = LDX(slot);
  rs = __fdiv_rn(amax, kRowScaleDiv);
  rinv = rs != 0.0f ? __frcp_rn(rs) : 0.0f;
}

// The 16 bf16 of block b of row (r, h): 32 bytes, 16-byte aligned.
__device__ __forceinline__ void load_block(const TensorNvfp4Params& p, uint32_t r, uint32_t h, uint32_t b,
                                           uint32_t (&w)[8]) {
  const uint16_t* src = p.x + static_cast<int64_t>(r) * p.row_pitch + static_cast<int64_t>(h) * p.head_pitch + 16 * b;
  uint32_t a[4], c[4];
  load16B(src, a);
  load16B(src + 8, c);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i] = a[i];
    w[4 + i] = c[i];
  }
}

// 1. amax of the tensor (every block of 16 of every row), into the scale slot.
__global__ void __launch_bounds__(kThreads) tensor_amax_kernel(const TensorNvfp4Params p) {
  const uint32_t nblk = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H) * static_cast<uint32_t>(p.D / 16);
  float m = 0.0f;
  for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < nblk; i += gridDim.x * kThreads) {
    uint32_t rh, b, r, h;
    p.div_nb.divmod(i, rh, b);
    p.div_h.divmod(rh, r, h);
    uint32_t w[8];
    load_block(p, r, h, b, w);
    m = fmaxf(m, absmax16(w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.rscale), __float_as_uint(m));
}

// 2a. VALUE kind: one thread per 16-channel block of a row.
__global__ void __launch_bounds__(kThreads) tensor_value_encode_kernel(const TensorNvfp4Params p) {
  const uint32_t nb = static_cast<uint32_t>(p.D / 16);
  const uint32_t nblk = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H) * nb;
  float rs, rinv;
  tensor_scale(p.rscale, rs, rinv);
  for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < nblk; i += gridDim.x * kThreads) {
    uint32_t rh, b, r, h;
    p.div_nb.divmod(i, rh, b);
    p.div_h.divmod(rh, r, h);
    uint32_t w[8];
    load_block(p, r, h, b, w);
    const uint32_t bsb = block_scale_code(absmax16(w), rs, rinv);
    uint32_t c0, c1;
    quantize_block(w, __fmul_rn(e4m3_to_f32(bsb), rs), c0, c1);
    store8B(p.codes + static_cast<int64_t>(rh) * (p.D / 2) + 8 * b, c0, c1);
    STX(p.bscale + static_cast<int64_t>(rh) * nb + b, static_cast<uint8_t>(bsb));
  }
}

// 2b. KEY kind: one thread per (group of 16 token rows, head, 8-channel chunk); the
// chunk's 8 blocks are its channels over the group's rows.  Each row is one 16-byte
// copy and one 4-byte code store; a partial group repeats its last row for the block
// maxima (no change to them) and stores only its own rows.  The rows arrive by
// cp.async in the thread's own shared-memory cells (row k at cell k * kThreads +
// thread, so a warp's reads are conflict-free); the next task's copies are issued
// once this task's cells have been read (the maxima use every read), so they travel
// while this task is coded.  The thread's own wait_group orders its cells.
constexpr size_t kKeySmem = static_cast<size_t>(16) * kThreads * 16;

__global__ void __launch_bounds__(kThreads, 2) tensor_key_encode_kernel(const TensorNvfp4Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint4* const cells = reinterpret_cast<uint4*>(smem) + threadIdx.x;
  const uint32_t nb = static_cast<uint32_t>(p.D / 16);  // chunk pairs per row
  const uint32_t ngroups = static_cast<uint32_t>((p.rows + 15) / 16);
  const uint32_t ntask = ngroups * static_cast<uint32_t>(p.H) * 2u * nb;
  const uint32_t stride = gridDim.x * kThreads;
  struct Task {
    uint32_t g, h, ch;
    int r0, n;
  };
  auto task_of = [&](uint32_t i) {
    Task t;
    uint32_t gh, cp2;
    p.div_nb.divmod(i >> 1, gh, cp2);  // task i = gh * D/8 + chunk
    p.div_h.divmod(gh, t.g, t.h);
    t.ch = 2u * cp2 + (i & 1u);
    t.r0 = static_cast<int>(t.g) * 16;
    t.n = min(16, p.rows - t.r0);
    return t;
  };
  auto issue = [&](uint32_t i) {
    if (i >= ntask) return;
    const Task t = task_of(i);
    const uint16_t* const src = p.x + static_cast<int64_t>(t.h) * p.head_pitch + 8 * t.ch;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      cp_async16(cells + k * kThreads, src + static_cast<int64_t>(t.r0 + min(k, t.n - 1)) * p.row_pitch);
  };
  float rs, rinv;
  tensor_scale(p.rscale, rs, rinv);
  uint32_t i = blockIdx.x * kThreads + threadIdx.x;
  issue(i);
  cp_async_commit();
  for (; i < ntask; i += stride) {
    cp_async_wait<0>();
    const Task t = task_of(i);
    uint32_t w[16][4];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 v = cells[k * kThreads];
      w[k][0] = v.x;
      w[k][1] = v.y;
      w[k][2] = v.z;
      w[k][3] = v.w;
    }
    // |max| of each channel over the 16 rows, as a pairwise tree (depth 4)
    uint32_t m[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t t[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = absmax2(w[2 * k][j], w[2 * k + 1][j]);
#pragma unroll
      for (int k = 0; k < 4; ++k) t[k] = absmax2(t[2 * k], t[2 * k + 1]);
      m[j] = absmax2(absmax2(t[0], t[1]), absmax2(t[2], t[3]));
    }
    issue(i + stride);  // every cell has been read (the maxima use them all)
    cp_async_commit();
    uint32_t bsc[8];
    float sc[8], inv[8];
    bool direct = false;  // a tiny scale: divide instead
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t mj = m[j] & 0x7FFF7FFFu;
      bsc[2 * j] = block_scale_code(bf16lo(mj), rs, rinv);
      bsc[2 * j + 1] = block_scale_code(bf16hi(mj), rs, rinv);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      sc[c] = __fmul_rn(e4m3_to_f32(bsc[c]), rs);
      inv[c] = sc[c] != 0.0f ? __frcp_rn(sc[c]) : 0.0f;
      direct = direct || isinf(inv[c]);
    }
    uint64_t inv2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) inv2[j] = pack_f32x2(__float_as_uint(inv[2 * j]), __float_as_uint(inv[2 * j + 1]));
    uint8_t* const cp = p.codes + (static_cast<int64_t>(t.r0) * p.H + t.h) * (p.D / 2) + 4 * t.ch;
    const int64_t cstride = static_cast<int64_t>(p.H) * (p.D / 2);
    if (!direct && t.n == 16) {  // a full group with ordinary scales: unrolled
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        uint32_t byte[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t a, b;
          unpack_f32x2(mul_f32x2(pack_f32x2(w[k][j] << 16, w[k][j] & 0xFFFF0000u), inv2[j]), a, b);
          byte[j] = e2m1x2_from_f32(__uint_as_float(a), __uint_as_float(b));
        }
        STX(reinterpret_cast<uint32_t*>(cp + k * cstride), bytes4(byte[0], byte[1], byte[2], byte[3]));
      }
    } else {  // a partial group, or a scale whose reciprocal overflows (divide): compact,
              // the rows read again from global memory (the cells hold the next task)
      const uint16_t* const src = p.x + static_cast<int64_t>(t.h) * p.head_pitch + 8 * t.ch;
#pragma unroll 1
      for (int k = 0; k < t.n; ++k) {
        uint32_t wk[4];
        load16B(src + static_cast<int64_t>(t.r0 + k) * p.row_pitch, wk);
        uint32_t byte[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float xl = bf16lo(wk[j]), xh = bf16hi(wk[j]);
          const float ql = isinf(inv[2 * j]) ? __fdiv_rn(xl, sc[2 * j]) : __fmul_rn(xl, inv[2 * j]);
          const float qh = isinf(inv[2 * j + 1]) ? __fdiv_rn(xh, sc[2 * j + 1]) : __fmul_rn(xh, inv[2 * j + 1]);
          byte[j] = e2m1x2_from_f32(ql, qh);
        }
        STX(reinterpret_cast<uint32_t*>(cp + k * cstride), bytes4(byte[0], byte[1], byte[2], byte[3]));
      }
    }
    store8B(p.bscale + (static_cast<int64_t>(t.g) * p.H + t.h) * p.D + 8 * t.ch,
            bytes4(bsc[0], bsc[1], bsc[2], bsc[3]), bytes4(bsc[4], bsc[5], bsc[6], bsc[7]));
  }
  cp_async_wait<0>();  // only empty groups remain; nothing is left in flight at exit
}

// 3. The scale slot: amax -> rs (the decode multiplier).
__global__ void tensor_scale_finalize_kernel(float* slot) {
  STX(slot, __fdiv_rn(LDX(slot), kRowScaleDiv));
}

// Unpack, KEY kind: one thread per 16 channels of a row; each channel has its own
// block scale (of the row's 16-row group).
__global__ void __launch_bounds__(kThreads) tensor_key_decode_kernel(const TensorNvfp4Params p) {
  const uint32_t nb = static_cast<uint32_t>(p.D / 16);
  const uint32_t nblk = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H) * nb;
  const float rs = LDX(p.rscale);
  const uint64_t rs2 = pack_f32x2(__float_as_uint(rs), __float_as_uint(rs));
  for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < nblk; i += gridDim.x * kThreads) {
    uint32_t rh, j, r, h;
    p.div_nb.divmod(i, rh, j);
    p.div_h.divmod(rh, r, h);
    uint32_t c0, c1, bsw[4];
    load8B(p.codes + static_cast<int64_t>(rh) * (p.D / 2) + 8 * j, c0, c1);
    load16B(p.bscale + (static_cast<int64_t>(r / 16) * p.H + h) * p.D + 16 * j, bsw);
    uint32_t out[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t byte = ((e < 4 ? c0 : c1) >> (8 * (e & 3))) & 0xFFu;
      const uint32_t h2 = e2m1x2_to_f16x2(byte);
      const uint32_t two = (bsw[e / 2] >> (16 * (e % 2))) & 0xFFFFu;  // scales of channels 2e, 2e + 1
      const float lo = mul_f16_to_f32(static_cast<uint16_t>(h2 & 0xFFFFu),
                                      static_cast<uint16_t>(e4m3_to_f16x2(two & 0xFFu) & 0xFFFFu));
      const float hi = mul_f16_to_f32(static_cast<uint16_t>(h2 >> 16),
                                      static_cast<uint16_t>(e4m3_to_f16x2(two >> 8) & 0xFFFFu));
      uint32_t yl, yh;
      unpack_f32x2(mul_f32x2(pack_f32x2(__float_as_uint(lo), __float_as_uint(hi)), rs2), yl, yh);
      out[e] = pack_bf16x2(__uint_as_float(yl), __uint_as_float(yh));
    }
    uint16_t* dst = p.y + static_cast<int64_t>(r) * p.y_row_pitch + static_cast<int64_t>(h) * p.y_head_pitch + 16 * j;
    store16B(dst, *reinterpret_cast<const uint32_t(*)[4]>(&out[0]));
    store16B(dst + 8, *reinterpret_cast<const uint32_t(*)[4]>(&out[4]));
  }
}

template <typename K>
int grid_for(K kernel, uint32_t work, size_t smem = 0) {
  const int occ = cached_occupancy(reinterpret_cast<const void*>(kernel), kThreads, smem);
  const int64_t need = (static_cast<int64_t>(work) + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * occ;
  return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

cudaError_t launch_tensor_nvfp4_pack(const TensorNvfp4Params& p, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.rscale, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  const uint32_t nblk = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H) * static_cast<uint32_t>(p.D / 16);
  KVQ_LAUNCH("tensor_amax_kernel", s,
             tensor_amax_kernel<<<grid_for(tensor_amax_kernel, nblk), kThreads, 0, s>>>(p); e = cudaGetLastError());
  if (e != cudaSuccess) return e;
  if (p.kind == 0) {
    const uint32_t ntask = static_cast<uint32_t>((p.rows + 15) / 16) * static_cast<uint32_t>(p.H) *
                           static_cast<uint32_t>(p.D / 8);
    e = cudaFuncSetAttribute(tensor_key_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kKeySmem));  // the shared-memory opt-in (per device)
    if (e != cudaSuccess) return e;
    KVQ_LAUNCH("tensor_key_encode_kernel", s,
               tensor_key_encode_kernel<<<grid_for(tensor_key_encode_kernel, ntask, kKeySmem), kThreads, kKeySmem, s>>>(p);
               e = cudaGetLastError());
  } else {
    KVQ_LAUNCH("tensor_value_encode_kernel", s,
               tensor_value_encode_kernel<<<grid_for(tensor_value_encode_kernel, nblk), kThreads, 0, s>>>(p);
               e = cudaGetLastError());
  }
  if (e != cudaSuccess) return e;
  KVQ_LAUNCH("tensor_scale_finalize_kernel", s,
             tensor_scale_finalize_kernel<<<1, 1, 0, s>>>(p.rscale); e = cudaGetLastError());
  return e;
}

// KEY kind only: V blocks run along channels, the row codec's layout with one scale for
// every row, and decode through the row-codec decode kernel.
cudaError_t launch_tensor_nvfp4_unpack(const TensorNvfp4Params& p, cudaStream_t s) {
  if (p.kind != 0) return cudaErrorInvalidValue;
  const uint32_t nblk = static_cast<uint32_t>(p.rows) * static_cast<uint32_t>(p.H) * static_cast<uint32_t>(p.D / 16);
  cudaError_t e = cudaSuccess;
  KVQ_LAUNCH("tensor_key_decode_kernel", s,
             tensor_key_decode_kernel<<<grid_for(tensor_key_decode_kernel, nblk), kThreads, 0, s>>>(p);
             e = cudaGetLastError());
  return e;
}

}  // namespace kvq
