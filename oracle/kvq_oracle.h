/*
 * kvq_oracle.h -- plain scalar CPU oracle for the KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the tests, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no source, header, table or constant with the
 * CUDA library; both are checked against each other on the same seeded inputs.
 *
 * Every floating-point step is one IEEE-754 binary32 operation with
 * round-to-nearest-even, in the order written in kvq_oracle.c.  Build with
 * -ffp-contract=off and without fast-math (no FTZ/DAZ).
 *
 * bf16 values are passed as their uint16 bit patterns, fp16 metadata likewise.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against facts the pages or the mathematics fix (format enumerations, the
 * e4m3 -> fp16 bit identity printed on the FreeToken page, exact round trips,
 * closed forms, brute force).  One property is NOT pinned: bit parity with
 * vLLM's ref_nvfp4_quant and FlashLoop's packing.py, whose source is not
 * available ("parity unpinned" for that comparison only).
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status bits the oracle reports for data-dependent faults (rows skipped). */
#define ORC_BAD_SLOT 1u    /* slot id >= number of slots */
#define ORC_BAD_BLOCK 2u   /* block-table entry outside the pool */
#define ORC_BAD_POS 4u     /* position out of [0, T) or not strictly increasing */
#define ORC_BAD_SEQLEN 8u  /* sequence length outside [0, min(Tmax, max_blocks*block_size)] */

enum { ORC_FMT_NVFP4 = 1, ORC_FMT_INT4 = 2, ORC_FMT_FP8 = 3, ORC_FMT_NVFP4_TENSOR = 4 };
enum { ORC_KIND_KEY = 0, ORC_KIND_VALUE = 1 };

/* 1 when this host's binary32 arithmetic keeps subnormal operands and results (no
 * flush-to-zero, no denormals-are-zero), else 0.  The oracle's definitions assume it;
 * the Python loader refuses to use the library when it returns 0. */
int orc_subnormals_kept(void);

/* ---- scalar format primitives ---- */
float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);
float orc_e2m1_value(uint8_t code);     /* signed nibble -> value */
uint8_t orc_e2m1_encode(float q);       /* sign of q | RNE magnitude code, saturating at 6 */
float orc_e4m3_value(uint8_t code);     /* byte -> value (NaN for 0x7F / 0xFF) */
uint8_t orc_e4m3_encode(float t);       /* RNE, saturating at +-448 */

/* Array forms of the primitives (for exhaustive pins from Python). */
void orc_f32_to_bf16_n(const float* x, int64_t n, uint16_t* y);
void orc_f32_to_f16_n(const float* x, int64_t n, uint16_t* y);
void orc_e2m1_encode_n(const float* x, int64_t n, uint8_t* y);
void orc_e4m3_encode_n(const float* x, int64_t n, uint8_t* y);

/* ---- NVFP4 row codec: one row of D bf16 (D % 16 == 0) ---- */
void orc_nvfp4_encode_row(const uint16_t* x, int D, uint8_t* codes, uint8_t* bscale,
                          float* rscale);
void orc_nvfp4_decode_row(const uint8_t* codes, const uint8_t* bscale, float rscale, int D,
                          uint16_t* y);
/* n contiguous rows: x [n][D] -> codes [n][D/2], bscale [n][D/16], rscale [n] */
void orc_nvfp4_encode_rows(const uint16_t* x, int64_t n, int D, uint8_t* codes,
                           uint8_t* bscale, float* rscale);
void orc_nvfp4_decode_rows(const uint8_t* codes, const uint8_t* bscale, const float* rscale,
                           int64_t n, int D, uint16_t* y);

/* ---- FP8 E4M3 row codec: one row of D bf16 -> D E4M3 codes + one FP32 scale ---- */
void orc_fp8_encode_row(const uint16_t* x, int D, uint8_t* codes, float* rscale);
void orc_fp8_decode_row(const uint8_t* codes, float rscale, int D, uint16_t* y);
void orc_fp8_encode_rows(const uint16_t* x, int64_t n, int D, uint8_t* codes, float* rscale);
void orc_fp8_decode_rows(const uint8_t* codes, const float* rscale, int64_t n, int D, uint16_t* y);

/* ---- paged store / restore (one tensor, K or V) ----
 * x is addressed x[t*row_pitch + h*head_pitch + d] (elements).
 * Pool planes: codes [num_slots][H][D/2], bscale [num_slots][H][D/16], rscale [num_slots][H].
 * slot_ids[t] < 0 means "skip"; >= num_slots sets ORC_BAD_SLOT and skips. */
uint32_t orc_nvfp4_scatter(const uint16_t* x, int64_t row_pitch, int64_t head_pitch, int T,
                           int H, int D, const int64_t* slot_ids, int64_t num_slots,
                           uint8_t* codes, uint8_t* bscale, float* rscale);
/* out [S][Tmax][H][D]; rows t >= seq_lens[s] are left untouched. */
uint32_t orc_nvfp4_restore(const uint8_t* codes, const uint8_t* bscale, const float* rscale,
                           int64_t num_slots, int H, int D, int block_size,
                           const int32_t* block_table, int S, int max_blocks,
                           const int32_t* seq_lens, int Tmax, uint16_t* out);
/* FP8 pool planes: codes [num_slots][H][D], rscale [num_slots][H]. */
uint32_t orc_fp8_scatter(const uint16_t* x, int64_t row_pitch, int64_t head_pitch, int T, int H,
                         int D, const int64_t* slot_ids, int64_t num_slots, uint8_t* codes,
                         float* rscale);
uint32_t orc_fp8_restore(const uint8_t* codes, const float* rscale, int64_t num_slots, int H,
                         int D, int block_size, const int32_t* block_table, int S,
                         int max_blocks, const int32_t* seq_lens, int Tmax, uint16_t* out);

/* ---- NVFP4 with one FP32 scale per tensor (vllm-rlt PR #166's logical layout) ----
 * x contiguous [T][H][D] (D % 16 == 0).  rs = amax over the whole tensor / 2688.
 * Blocks of 16 run along the kind's axis: kind VALUE over 16 channels per (t, h),
 * kind KEY over 16 token rows per (h, d) (the last group may be partial).  Per block
 * the row codec's steps R2-R3 against the tensor's rs.  Layout:
 *   codes [T][H][D/2] (low nibble = even channel)
 *   bscale: VALUE [T][H][D/16], KEY [ceil(T/16)][H][D]
 *   rscale [1] */
void orc_nvfp4t_pack(const uint16_t* x, int T, int H, int D, int kind, uint8_t* codes,
                     uint8_t* bscale, float* rscale);
void orc_nvfp4t_unpack(const uint8_t* codes, const uint8_t* bscale, const float* rscale, int T, int H,
                       int D, int kind, uint16_t* y);

/* ---- INT4 affine codec, group size G, x contiguous [T][H][D] (D even) ----
 * codes [T][H][D/2] (low nibble = even channel)
 * key:   groups of G token rows per (h, d): mn16/sc16 [ceil(T/G)][H][D]
 * value: groups of G channels per (t, h):   mn16/sc16 [T][H][ceil(D/G)] */
void orc_int4_pack(const uint16_t* x, int T, int H, int D, int kind, int G, uint8_t* codes,
                   uint16_t* mn16, uint16_t* sc16);
void orc_int4_unpack(const uint8_t* codes, const uint16_t* mn16, const uint16_t* sc16, int T,
                     int H, int D, int kind, int G, uint16_t* y);

/* ---- residual encode / decode ----
 * cur, prev, out: contiguous [T][H][D].  pos: P strictly increasing positions in [0, T), or
 * NULL for the dense case (P must equal T).  The payload covers the P compact rows:
 *   NVFP4: codes [P][H][D/2], meta_a = bscale [P][H][D/16] (uint8), rscale [P][H]
 *   INT4 : codes [P][H][D/2], meta_a = mn16, meta_b = sc16 (uint16, shapes as orc_int4_pack)
 *   FP8  : codes [P][H][D], rscale [P][H]
 * pos_out receives the owned copy of the positions (may be NULL when pos is NULL). */
uint32_t orc_residual_encode(const uint16_t* cur, const uint16_t* prev, int T, int H, int D,
                             const int32_t* pos, int P, int fmt, int kind, int G,
                             uint8_t* codes, void* meta_a, void* meta_b, float* rscale,
                             int32_t* pos_out);
uint32_t orc_residual_decode(const uint8_t* codes, const void* meta_a, const void* meta_b,
                             const float* rscale, int fmt, int kind, int G, const int32_t* pos,
                             int P, const uint16_t* prev, int T, int H, int D, uint16_t* out);

/* ---- paged decode attention over a quantised pool (fp64) ----
 * One query token per sequence.  Query head qh reads KV head qh / (Hq / H) (Hq a
 * multiple of H).  K and V rows are the exact decoded values: NVFP4 e2m1 * bs * rs,
 * FP8 e4m3 * rs (fmt_k / fmt_v per plane; bscale NULL for FP8).  For every sequence s
 * with 0 < len = seq_lens[s]:
 *   s_t = scale * sum_d q[s][qh][d] * k[t][d],  p = softmax_t(s),  out = sum_t p_t v[t]
 * over tokens t < len (slot = block_table[s][t / block_size] * block_size + t % block_size).
 * len == 0 writes zeros.  A bad length, or a block entry outside the pool, flags the
 * status and leaves that sequence's output untouched.
 * q: bf16 bits [S][Hq][D]; out: double [S][Hq][D]. */
uint32_t orc_decode_attention(const uint8_t* k_codes, const uint8_t* k_bscale, const float* k_rscale,
                              int fmt_k, const uint8_t* v_codes, const uint8_t* v_bscale,
                              const float* v_rscale, int fmt_v, int64_t num_slots, int H, int D,
                              int block_size, const int32_t* block_table, int S, int max_blocks,
                              const int32_t* seq_lens, const uint16_t* q, int Hq, double scale,
                              double* out);

/* ---- storage accounting (bytes held by the codes and their scale sidecars) ---- */
int64_t orc_storage_bytes(int fmt, int kind, int G, int64_t T, int H, int D);

#ifdef __cplusplus
}
#endif
#endif
