// kvq_params.h -- launch parameter blocks passed by value from the C ABI layer to
// the kernels, and the host-side launch functions each kernel file defines.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// Exact unsigned division of n < 2^31 by a fixed divisor d >= 1 with one
// multiply-high, an add and a shift (Granlund & Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, the round-up method):
//   l = ceil(log2 d),  m = floor(2^32 * (2^l - d) / d) + 1,
//   n / d = (mulhi(m, n) + n) >> l.
// For n < 2^31 the sum cannot overflow 32 bits.
struct FastDiv {
  uint32_t d = 1, m = 0, l = 0;
  FastDiv() = default;
  __host__ __device__ explicit FastDiv(uint32_t div) : d(div) {
    l = 0;
    while ((1ull << l) < div) ++l;
    uint64_t two_l = 1ull << l;
    m = static_cast<uint32_t>(((two_l - div) << 32) / div + 1);
  }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    uint32_t hi = __umulhi(m, n);
#else
    uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(m) * n) >> 32);
#endif
    return (hi + n) >> l;
  }
  __host__ __device__ __forceinline__ void divmod(uint32_t n, uint32_t& q, uint32_t& r) const {
    q = div(n);
    r = n - q * d;
  }
};

// ---------------------------------------------------------------------------
// NVFP4 encode: quant-scatter, logical pack and residual encode share one kernel.
// ---------------------------------------------------------------------------
enum EncodeMode : int { kEncScatter = 0, kEncPack = 1, kEncResidual = 2 };

struct Nvfp4Planes {
  uint8_t* codes;   // NVFP4 [rows][D/2], FP8 [rows][D]  (rows = slot*H + h, or p*H + h)
  uint8_t* bscale;  // NVFP4 [rows][D/16]
  float* rscale;    // [rows]
};

struct EncodeTensor {
  const uint16_t* x;     // bf16 source (residual: current)
  int64_t row_pitch;     // elements
  int64_t head_pitch;
  const uint16_t* prev;  // residual: reconstructed predecessor
  int64_t prev_row_pitch;
  int64_t prev_head_pitch;
  Nvfp4Planes dst;
};

struct EncodeParams {
  EncodeTensor ten[2];
  int32_t ntensors;         // 1 or 2
  uint32_t rows_per_tensor; // tokens * H (residual: num_pos * H)
  FastDiv div_h;            // by H
  int32_t H;
  int32_t nb;               // D / 16
  const int64_t* slot_ids;  // scatter
  int64_t num_slots;
  const int32_t* pos;       // residual; nullptr = dense
  int32_t* pos_out;
  int32_t src_rows;         // residual: rows of cur/prev (positions must be below)
  uint32_t* status;
};

// ---------------------------------------------------------------------------
// NVFP4 decode: paged restore and logical unpack.
// ---------------------------------------------------------------------------
enum DecodeMode : int { kDecRestore = 0, kDecUnpack = 1 };

struct DecodeTensor {
  const uint8_t* codes;
  const uint8_t* bscale;
  const float* rscale;
  uint16_t* y;
  int64_t row_pitch;
  int64_t head_pitch;
};

struct DecodeParams {
  DecodeTensor ten[2];
  int32_t ntensors;
  uint32_t rows_per_tensor;  // restore: S * Tmax * H; unpack: rows * H
  FastDiv div_h;             // by H
  FastDiv div_tmax;          // by Tmax (restore)
  FastDiv div_bs;            // by block_size (restore)
  int32_t H;
  int32_t nb;
  const int32_t* block_table;  // [S][max_blocks]
  const int32_t* seq_lens;     // [S]
  int32_t max_blocks;
  int32_t tmax;
  int32_t seq_cap;             // min(Tmax, max_blocks * block_size)
  int64_t num_blocks;
  int32_t block_size;
  uint32_t* status;
};

// ---------------------------------------------------------------------------
// INT4 affine codec and residual decode.
// ---------------------------------------------------------------------------
struct Int4Payload {
  uint8_t* codes;   // [rows][H][D/2]
  uint16_t* mn;     // fp16 bits
  uint16_t* sc;     // fp16 bits
};

struct Int4EncodeParams {
  const uint16_t* x;  // residual: current
  int64_t row_pitch, head_pitch;
  const uint16_t* prev;
  int64_t prev_row_pitch, prev_head_pitch;
  Int4Payload dst;
  int32_t rows;       // compact rows (T, or num_pos)
  FastDiv div_h;      // by H
  int32_t H, D, G;
  int32_t kind;       // 0 key, 1 value
  int32_t residual;   // 0/1
  const int32_t* pos;
  int32_t* pos_out;
  int32_t src_rows;
  uint32_t* status;
};

// Decoder of a packed payload row into bf16, plus an optional residual add.
struct PayloadRef {
  int32_t fmt;         // 1 nvfp4, 2 int4, 3 fp8
  int32_t kind;
  int32_t G;
  const uint8_t* codes;
  const void* meta0;   // nvfp4: bscale; int4: min
  const void* meta1;   // int4: scale
  const float* rscale; // nvfp4 / fp8: row scale of row r at rscale[r * rs_stride]
  int32_t rs_stride;   // 1 (one scale per row), or 0 (one scale for the whole tensor)
  int32_t rows;
};

struct UnpackParams {
  PayloadRef pay;
  int32_t H, D, nb;
  FastDiv div_h;
  uint32_t total_rows;  // rows * H of the iteration space
  // plain unpack: y = decode(payload)
  uint16_t* y;
  int64_t y_row_pitch, y_head_pitch;
  // residual decode: out = prev (+ decode at kept rows)
  const uint16_t* prev;
  int64_t prev_row_pitch, prev_head_pitch;
  const int32_t* pos;   // nullptr = dense
  int32_t num_pos;
  int32_t src_rows;     // rows of prev/out
  int32_t mode;         // 0 unpack, 1 residual in place (iterate kept rows), 2 residual out of place
  int32_t run;          // residual copy: tokens per warp run (set by the launcher)
  uint32_t* status;
};

// Checked build only: the byte ranges a launch may touch, registered by the C ABI
// layer before each launch and copied to the device by the launcher.
namespace dbg {
struct HostRange {
  unsigned long long lo, hi;
  const char* name;
};
HostRange* pending(int* n);  // the list for the next launch (at most 32 entries)
}  // namespace dbg

// Launchers (return the cudaGetLastError() of the launch).  fmt: 1 NVFP4, 3 FP8.
cudaError_t launch_nvfp4_encode(const EncodeParams& p, int mode, int fmt, bool v8,
                                cudaStream_t s);
cudaError_t launch_nvfp4_decode(const DecodeParams& p, int mode, int fmt, bool v8,
                                cudaStream_t s);
cudaError_t launch_int4_encode(const Int4EncodeParams& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// NVFP4 with one FP32 scale per tensor (logical pack / unpack).
// ---------------------------------------------------------------------------
struct TensorNvfp4Params {
  const uint16_t* x;        // pack source [rows][H][D] through the pitches
  int64_t row_pitch, head_pitch;
  uint8_t* codes;           // [rows][H][D/2]
  uint8_t* bscale;          // KEY [ceil(rows/16)][H][D], VALUE [rows][H][D/16]
  float* rscale;            // [1]
  uint16_t* y;              // unpack output through its pitches
  int64_t y_row_pitch, y_head_pitch;
  int32_t rows, H, D, kind;
  FastDiv div_h;            // by H
  FastDiv div_nb;           // by D/16
  FastDiv div_np;           // by D/2
};

cudaError_t launch_tensor_nvfp4_pack(const TensorNvfp4Params& p, cudaStream_t s);
cudaError_t launch_tensor_nvfp4_unpack(const TensorNvfp4Params& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// Paged decode attention over the quantised pool.
// ---------------------------------------------------------------------------
struct AttnPlane {
  const uint8_t* codes;   // [slots][H][D/2] (NVFP4) or [slots][H][D] (FP8)
  const uint8_t* bscale;  // [slots][H][D/16] (NVFP4)
  const float* rscale;    // [slots][H]
};

struct AttnParams {
  AttnPlane k, v;
  int32_t fmt_k, fmt_v;
  const uint16_t* q;        // bf16 [S][Hq][D] through the pitches below
  int64_t q_row_pitch, q_head_pitch;
  uint16_t* out;            // bf16, same indexing through its own pitches
  int64_t o_row_pitch, o_head_pitch;
  float* ws;                // split partials [S][Hq][nsplit][D + 2] (nsplit > 1)
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t max_blocks;
  int32_t seq_cap;          // max_blocks * block_size
  int32_t block_size;
  FastDiv div_bs;
  int64_t num_blocks;
  int32_t S, H, Hq, D, group;  // group = Hq / H query heads per KV head
  int32_t max_len;          // max_seq_len of the call (the split policy's input)
  int32_t nsplit;           // set by the launch: token splits per sequence
  int32_t split_len;        // set by the launch: tokens per split
  float scale;              // softmax scale applied to q . k
  uint32_t* status;
};

// Split count of the head-major kernel: enough CTAs to fill the GPU, each split at
// least 256 tokens.
int attn_num_splits(int32_t S, int32_t H, int32_t max_seq_len);
// Workspace bytes for the split partials of a call, whichever kernel serves it.
size_t attn_workspace_bytes(int32_t S, int32_t H, int32_t Hq, int32_t D, int32_t max_seq_len);
cudaError_t launch_decode_attention(const AttnParams& p, cudaStream_t s);
// The library's built-in split scratch (device memory in the library image, for the
// entry point that allocates nothing): its device address and size in bytes.
cudaError_t attn_builtin_scratch(void** ptr, size_t* bytes);
size_t attn_builtin_scratch_bytes();
cudaError_t launch_payload_decode(const UnpackParams& p, int lanes, bool v8, cudaStream_t s);

int num_sms();

// Resident blocks per SM of a kernel at a block size and dynamic shared memory, on the
// current device; queried once per (kernel, block size, shared memory, device) and
// kept, so eager calls do not repeat the occupancy query.  At least 1.
int cached_occupancy(const void* kernel, int threads, size_t smem);

}  // namespace kvq
