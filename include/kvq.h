/*
 * kvq.h -- C ABI of the GB300 KV-cache quantisation codec (libkvq.so).
 *
 * The library turns bf16 K/V rows into compact KV-cache formats and back, with
 * hand-written sm_103a CUDA kernels:
 *   - NVFP4 row codec: per (token, KV head) row of head_dim values, packed E2M1
 *     nibbles (low nibble = even element), an E4M3 scale for each block of 16 and
 *     an FP32 scale for the row: head_dim/2 + head_dim/16 + 4 bytes (76 B at head_dim 128).
 *     Source: "feat(kvcache): add nvfp4 kv quantization (FreeToken PR #408)",
 *     Summary and the codec-delta port note.
 *   - INT4 affine codec with group size G (G64 by default), FP32 arithmetic and
 *     FP16 min/scale metadata; K grouped over token rows per (head, channel), V
 *     over channels per (token, head).  Source: "vllm-rlt PR #166: INT4 KV
 *     packing/unpacking and cross-loop residual reconstruction", Purpose.
 *   - Residual encode/decode against the reconstructed predecessor with a compact
 *     int32 position map (same page, Purpose).
 *   - FP8 E4M3 row codec: one E4M3 byte per element and a single FP32 scale for
 *     each (token, KV head) row, in a code buffer with the geometry of the bf16 one.
 *     Source: FreeToken PR #408, the fp8 store notes.
 *
 * Conventions shared by every entry point
 *   Memory   every pointer argument that a kernel touches is DEVICE memory
 *            (cudaMalloc / the torch caching allocator) owned by the caller.  The
 *            library allocates nothing, frees nothing and never synchronises, so
 *            every entry point but kvq_decode_attention_noalloc (see there) may be
 *            captured in a CUDA graph.  Host or unregistered
 *            pointers are rejected with KVQ_ERR_NOT_DEVICE_PTR before any launch
 *            (the FreeToken page records a host tensor handed to a kernel).
 *   bf16     K/V tensors are bf16 [rows][heads][dim] views with inner stride 1 and
 *            their OWN row and head pitches, in elements.  K and V never share a
 *            pitch argument: the FreeToken page records a store kernel that read V
 *            at K's row pitch and corrupted it.
 *   Streams  work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   Errors   argument errors are returned as kvq_status before anything is
 *            launched; kvq_last_error() gives a one-line reason (thread-local).
 *            Data-dependent errors (a slot id past the pool, a block-table entry
 *            outside the pool, a bad position) can only be seen on the device: the
 *            kernel skips the offending row and ORs a KVQ_DEV_* bit into
 *            *dev_status (a caller-owned device uint32, may be NULL).  No kernel
 *            traps or asserts, so a bad id never poisons the CUDA context (the
 *            FreeToken page records a device-side assert that did).
 *   Floats   every result is bit-exact against the plain CPU definition of the
 *            codec: one IEEE binary32 operation at a time, round to nearest even,
 *            no FMA contraction, no flush to zero, in this order.  NVFP4 encode:
 *            rs = amax / 2688; per 16-block t = min((vb / 6) / rs, 448) (0 if rs is
 *            0), bs = E4M3(t), s = bs * rs, q = x * (1 / s) (x / s when 1 / s
 *            overflows, signed zeros when s is 0), code = E2M1(min(|q|, 6)) with
 *            x's sign.  NVFP4 decode: bf16((e2m1 * bs) * rs).  FP8: rs = amax / 448,
 *            q = x * (1 / rs), decode bf16(e4m3 * rs).  INT4: sc = (mx - mn) / 15,
 *            code = clamp(rint((x - mn) / sc), 0, 15) from the FP32 mn and sc (codes
 *            0 when sc is 0), then FP16 metadata; decode bf16(code * sc16 + mn16).
 *            Residuals: r = bf16(cur - prev), out = bf16(prev + decoded r).
 *   Inputs   finite values only; INT4 also needs |x| < 65504 (FP16 metadata).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

typedef struct CUstream_st* kvq_stream_t; /* identical to cudaStream_t */

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,    /* null/negative/inconsistent sizes or pointers */
  KVQ_ERR_UNSUPPORTED = 2,    /* a valid request this build does not implement */
  KVQ_ERR_MISALIGNED = 3,     /* a base or pitch breaks the 16-byte rule below */
  KVQ_ERR_NOT_DEVICE_PTR = 4, /* a pointer is host, unregistered or managed memory */
  KVQ_ERR_CUDA = 5            /* the CUDA runtime reported an error at launch */
} kvq_status;

typedef enum {
  KVQ_FMT_NVFP4 = 1,        /* row codec: E2M1 + E4M3 per 16 + one FP32 scale per row */
  KVQ_FMT_INT4 = 2,         /* affine INT4, FP16 minimum and scale per group of G */
  KVQ_FMT_FP8 = 3,          /* E4M3 + one FP32 scale per row */
  KVQ_FMT_NVFP4_TENSOR = 4  /* E2M1 + E4M3 per 16 along the kind's axis + one FP32 scale per tensor */
} kvq_format;
typedef enum { KVQ_KIND_KEY = 0, KVQ_KIND_VALUE = 1 } kvq_kind;

/* Bits ORed into *dev_status by the kernels. */
#define KVQ_DEV_BAD_SLOT 1u   /* slot id >= num_slots (row skipped) */
#define KVQ_DEV_BAD_BLOCK 2u  /* block-table entry < 0 or past the pool (row skipped) */
#define KVQ_DEV_BAD_POS 4u    /* position outside [0, rows) or not strictly increasing */
#define KVQ_DEV_BAD_SEQLEN 8u /* seq_lens[s] outside [0, min(max_seq_len, blocks*block_size)] */
#define KVQ_DEV_TIMEOUT 16u   /* decode attention: a bounded wait for a copy ran out (results unspecified) */

/* A bf16 view: element (r, h, d) is ptr[r*row_pitch + h*head_pitch + d].
 * ptr must be 16-byte aligned and both pitches multiples of 8 elements. */
typedef struct {
  const void* ptr;
  int64_t row_pitch;
  int64_t head_pitch;
} kvq_bf16_in;

typedef struct {
  void* ptr;
  int64_t row_pitch;
  int64_t head_pitch;
} kvq_bf16_out;

/* One tensor's planes in a paged pool, slot-major.  Format NVFP4:
 *   codes  [num_slots][num_heads][head_dim/2]   E2M1 nibbles, low nibble = even element
 *   bscale [num_slots][num_heads][head_dim/16]  E4M3 block scales
 *   rscale [num_slots][num_heads]               FP32 row scales
 * Format FP8: codes [num_slots][num_heads][head_dim] E4M3 bytes, rscale as above,
 * bscale unused (may be NULL).
 * Slot = block * block_size + offset.  Every plane used must be 16-byte aligned. */
typedef struct {
  uint8_t* codes;
  uint8_t* bscale;
  float* rscale;
} kvq_plane;

typedef struct {
  kvq_plane k;
  kvq_plane v;
  int64_t num_slots;  /* a multiple of block_size */
  int32_t block_size; /* tokens per page (16 in the pages' pools) */
  int32_t num_heads;
  int32_t head_dim;   /* a multiple of 16, at most 512 */
  int32_t fmt;        /* format of the K plane: KVQ_FMT_NVFP4 or KVQ_FMT_FP8 */
  int32_t v_fmt;      /* format of the V plane; 0 = the same as fmt.  FP8 K with NVFP4 V
                         is the k8v4 split of the FreeToken page (fp8 store notes) */
} kvq_pool;

/* A logical (non-paged) packed tensor [rows][heads][dim], caller-allocated.
 *   fmt NVFP4: codes [rows][heads][dim/2], meta0 = bscale uint8 [rows][heads][dim/16],
 *              rscale float [rows][heads], meta1 unused; group_size must be 16.
 *   fmt FP8  : codes [rows][heads][dim] E4M3, rscale float [rows][heads]; meta0 and
 *              meta1 unused; group_size ignored.
 *   fmt NVFP4_TENSOR: the logical NVFP4 layout of vllm-rlt PR #166 (Purpose): codes
 *              [rows][heads][dim/2], meta0 = bscale uint8, [ceil(rows/16)][heads][dim]
 *              for kind KEY (16 token rows per head and channel) or [rows][heads][dim/16]
 *              for kind VALUE (16 channels), rscale float [1] = tensor amax / 2688;
 *              group_size 16.  Logical pack / unpack only.
 *   fmt INT4 : codes [rows][heads][dim/2], meta0 = FP16 minimum, meta1 = FP16 scale,
 *              each [ceil(rows/G)][heads][dim] for kind KEY (groups of G token rows
 *              per head and channel) or [rows][heads][ceil(dim/G)] for kind VALUE
 *              (groups of G channels per token and head); rscale unused.
 *              G is one of 16, 32, 64, 128, 256, 512; the last group may be partial.
 * dim must be a multiple of 16 (at most 512); pointers 16-byte aligned. */
typedef struct {
  int32_t fmt;
  int32_t kind;
  int32_t group_size;
  int32_t rows;
  int32_t heads;
  int32_t dim;
  uint8_t* codes;
  void* meta0;
  void* meta1;
  float* rscale;
} kvq_packed;

/* Fused quantise + scatter of K and V into a paged pool (the encode hot path), each
 * in its plane's format (NVFP4, or FP8 E4M3 with one FP32 scale per row).
 * Source: FreeToken PR #408, Summary ("CUDA Graph-safe KV writes") and the fp8 store
 * notes (the destination slots are read from a device tensor; one launch under graph capture).
 *   k, v       bf16 [num_tokens][num_heads][head_dim] views; either may be NULL
 *              (that tensor is not stored); not both.
 *   slot_ids   device int64 [num_tokens]; token t goes to slot slot_ids[t]; a
 *              negative id skips the token (padding); an id >= num_slots skips it
 *              and sets KVQ_DEV_BAD_SLOT.  Duplicate ids: undefined last writer.
 *   pool       planes written in place (only the rows of the given slots).
 * One kernel launch (two when K and V planes have different formats); num_tokens ==
 * 0 launches nothing. */
KVQ_API kvq_status kvq_quant_scatter(const kvq_bf16_in* k, const kvq_bf16_in* v, int32_t num_tokens,
                             const int64_t* slot_ids, const kvq_pool* pool,
                             uint32_t* dev_status, kvq_stream_t stream);

/* Paged restore: gather and dequantise pool rows back to bf16 (the decode side).  Source: FreeToken PR #408, Summary ("Triton restore paths"); vllm-rlt
 * PR #166 review (pack_paged / unpack_paged over [pages, page_size, heads, dim]).
 *   block_table  device int32 [num_seqs][max_blocks]; token t of sequence s lives in
 *                slot block_table[s][t / block_size] * block_size + t % block_size.
 *   seq_lens     device int32 [num_seqs]; tokens t >= seq_lens[s] are not written.
 *   k_out/v_out  bf16 views of [num_seqs * max_seq_len][num_heads][head_dim]: row
 *                s * max_seq_len + t receives token t of sequence s.  Either may be
 *                NULL (that tensor is not restored); not both.
 * NVFP4: y = bf16(e2m1 * block_scale * row_scale), the product rounded once in fp32;
 * FP8: y = bf16(e4m3 * row_scale).  One launch (two when K and V planes have
 * different formats).
 * Rows with a bad block id are skipped (KVQ_DEV_BAD_BLOCK); a sequence with a bad
 * length is skipped whole (KVQ_DEV_BAD_SEQLEN). */
KVQ_API kvq_status kvq_restore(const kvq_pool* pool, const int32_t* block_table, int32_t num_seqs,
                       int32_t max_blocks, const int32_t* seq_lens, int32_t max_seq_len,
                       const kvq_bf16_out* k_out, const kvq_bf16_out* v_out,
                       uint32_t* dev_status, kvq_stream_t stream);

/* Logical pack: x [out->rows][out->heads][out->dim] -> *out in out->fmt / kind / G.
 * Source: vllm-rlt PR #166, Purpose (pack_kv(values, kind, format)). */
KVQ_API kvq_status kvq_pack(const kvq_bf16_in* x, const kvq_packed* out, kvq_stream_t stream);

/* Logical unpack: *in -> y [in->rows][in->heads][in->dim] bf16.
 * Source: vllm-rlt PR #166, Purpose (unpack_kv(packed)).
 * INT4: y = bf16(code * scale16 + min16), a mul then an add in fp32. */
KVQ_API kvq_status kvq_unpack(const kvq_packed* in, const kvq_bf16_out* y, kvq_stream_t stream);

/* Residual encode against the reconstructed predecessor.
 * Source: vllm-rlt PR #166, Purpose (encode_residual(current, previous, kind,
 * format); the kept rows are packed together, each call owning its int32 position list).
 *   cur, prev   bf16 [num_rows][heads][dim] (heads/dim from payload).
 *   pos         device int32 [num_pos], strictly increasing in [0, num_rows), or
 *               NULL for the dense case (then num_pos must equal num_rows).
 *   payload     packed [num_pos][heads][dim]: r[p] = bf16(cur[pos[p]] - prev[pos[p]])
 *               encoded in payload->fmt / kind / G (INT4 KEY groups follow the
 *               compact row order).  payload->rows must equal num_pos.
 *   pos_out     device int32 [num_pos] receiving the owned copy of pos (NULL: none).
 * A position outside [0, num_rows) contributes a zero residual row and sets
 * KVQ_DEV_BAD_POS; an unsorted map sets KVQ_DEV_BAD_POS (results then unspecified,
 * never out of bounds). */
KVQ_API kvq_status kvq_encode_residual(const kvq_bf16_in* cur, const kvq_bf16_in* prev,
                               int32_t num_rows, const int32_t* pos, int32_t num_pos,
                               const kvq_packed* payload, int32_t* pos_out,
                               uint32_t* dev_status, kvq_stream_t stream);

/* Residual decode: out = prev, and for every kept row p,
 * out[pos[p]] = bf16(prev[pos[p]] + unpack(payload)[p]).  Absent rows inherit prev.
 * Source: vllm-rlt PR #166, Purpose (decode_residual(residual, previous)).
 *   out  may be exactly prev (same pointer and pitches: in-place, only the kept rows
 *        are touched) or must not overlap it (every row is written).
 * Bad positions: as kvq_encode_residual (rows outside [0, num_rows) are skipped). */
KVQ_API kvq_status kvq_decode_residual(const kvq_packed* payload, const int32_t* pos, int32_t num_pos,
                               const kvq_bf16_in* prev, int32_t num_rows,
                               const kvq_bf16_out* out, uint32_t* dev_status,
                               kvq_stream_t stream);

/* Paged decode attention over a quantised pool: the step downstream of the
 * restore, with K and V dequantised in registers instead of restored to bf16.
 * Source: FreeToken PR #408, Summary (restore paths) and fp8 store notes (the row
 * scale multiplies the score and the output); vllm-rlt PR #166, review by 0z5a
 * (dequantise to 16 bits in registers and keep the 16-bit MMA).
 * One query token per sequence.  For query head qh (KV head qh / (num_q_heads /
 * pool->num_heads)):
 *   out[s][qh] = softmax_t(scale * q[s][qh] . k_t) . v_t   over t < seq_lens[s],
 * with k_t, v_t the decoded pool rows (each plane in its own format, NVFP4 or FP8).
 *   q    bf16 [num_seqs][num_q_heads][head_dim] through q->row_pitch (per sequence)
 *        and q->head_pitch (per head), inner stride 1; 16-byte aligned.
 *   out  bf16, indexed the same way through its own pitches.
 *   head_dim 64, 128 or 256; num_q_heads a multiple of num_heads, at most 16 query
 *   heads per KV head.  seq_lens[s] <= min(max_seq_len, max_blocks * block_size).
 *   scale  positive and finite (KVQ_ERR_INVALID_ARG otherwise).
 *   workspace  device memory of kvq_decode_attention_workspace(...) bytes, 16-byte
 *              aligned (may be NULL when that is 0); caller-owned, reused by the next
 *              call on the same stream.
 * Accuracy: K, V and Q enter the f16 MMA exactly (Q through a power-of-two
 * prescale); products and sums are fp32; P is rounded once to f16 (relative 2^-11,
 * relative to a reference of V's row scales) and the output once to bf16, so
 * |out - exact| <= 2^-9 |exact| + 2^-11 max|v| plus fp32 rounding, where exact is
 * the attention of the decoded rows.
 * An empty sequence writes zeros.  A bad length (KVQ_DEV_BAD_SEQLEN) or a block
 * entry outside the pool (KVQ_DEV_BAD_BLOCK) leaves that sequence's output untouched.
 * Every wait of the kernel on a copy into shared memory is bounded (about 0.1 s); one
 * that runs out sets KVQ_DEV_TIMEOUT, and the call's results are then unspecified.
 * One or two kernel launches. */
KVQ_API kvq_status kvq_decode_attention(const kvq_pool* pool, const int32_t* block_table,
                                        int32_t num_seqs, int32_t max_blocks, const int32_t* seq_lens,
                                        int32_t max_seq_len, const kvq_bf16_in* q, int32_t num_q_heads,
                                        float scale, const kvq_bf16_out* out, void* workspace,
                                        size_t workspace_bytes, uint32_t* dev_status,
                                        kvq_stream_t stream);

/* kvq_decode_attention for callers that cannot allocate device memory.  Some callers
 * have no way to hand the library a workspace: an engine whose memory planner has
 * already given all free HBM to the KV pool, or a host runtime that passes in only
 * the tensors it owns and offers no allocator hook.  A cudaMalloc can also
 * synchronise the device, which a decode step cannot afford.  This entry point
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine): the
 * split partials go to a scratch array that is part of the library image, 48 MiB of
 * device memory that every GPU which loads the library holds until the process exits.
 * The pages have no counterpart to this entry point; it exists for such callers.
 *   Limit    the partials need kvq_decode_attention_workspace(...) bytes; a call
 *            that needs more than 48 MiB returns KVQ_ERR_UNSUPPORTED.  The split
 *            policy keeps every supported shape under 40.2 MB on a 152-SM GPU.
 *   Set-up   the first call on a device looks up the scratch array's device address
 *            (with that device current) and keeps it; make that first call before
 *            any stream capture.  A failed lookup returns KVQ_ERR_CUDA.
 *   Sharing  there is one scratch array per device, shared by every call of this
 *            entry point on it, and it keeps the last call's contents (each call
 *            writes every partial it later reads, so nothing needs clearing).  Calls
 *            that overlap on the GPU race on it; kvq_decode_attention with a caller
 *            workspace has no such limit.
 * Arguments, argument checks, results and device status are those of
 * kvq_decode_attention without the workspace pair. */
KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_pool* pool, const int32_t* block_table,
                                                int32_t num_seqs, int32_t max_blocks,
                                                const int32_t* seq_lens, int32_t max_seq_len,
                                                const kvq_bf16_in* q, int32_t num_q_heads, float scale,
                                                const kvq_bf16_out* out, uint32_t* dev_status,
                                                kvq_stream_t stream);

/* Workspace bytes kvq_decode_attention needs for these sizes on the current device
 * (0 when the call runs without one).  Host-only query. */
KVQ_API size_t kvq_decode_attention_workspace(int32_t num_seqs, int32_t num_heads, int32_t num_q_heads,
                                              int32_t head_dim, int32_t max_seq_len);

/* Bytes held by codes plus scale sidecars for rows x heads x dim in a format,
 * excluding allocator overhead (vllm-rlt PR #166 review: storage_bytes).  76 per
 * NVFP4 row at dim 128; INT4 G64: 4 + 32/64 bits per element for full groups.
 * Returns 0 for an invalid request.  Host-only; needs no GPU. */
KVQ_API size_t kvq_storage_bytes(kvq_format fmt, kvq_kind kind, int32_t group_size, int64_t rows,
                         int32_t heads, int32_t dim);

/* Static name of a status code.  Host-only. */
KVQ_API const char* kvq_status_string(kvq_status status);

/* One-line reason for the last non-OK status returned on this thread. */
KVQ_API const char* kvq_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
