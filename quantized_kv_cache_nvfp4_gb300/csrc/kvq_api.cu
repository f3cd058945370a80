// kvq_api.cu -- the C ABI declared in include/kvq.h: argument checks on the host,
// then one kernel launch on the caller's stream.  Nothing here allocates, frees or
// synchronises, so every entry point can be captured in a CUDA graph.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kvq.h"
#include "kvq_params.h"

namespace kvq {

namespace {

thread_local char g_last_error[256] = "";

kvq_status fail(kvq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

// Checked build: the byte ranges of the next launch (see kvq_device.cuh).
thread_local dbg::HostRange g_ranges[32];
thread_local int g_nranges = 0;

void dbg_clear() { g_nranges = 0; }
void dbg_add(const void* p, int64_t bytes, const char* name) {
  if (p == nullptr || bytes <= 0 || g_nranges >= 32) return;
  const unsigned long long lo = reinterpret_cast<unsigned long long>(p);
  g_ranges[g_nranges++] = dbg::HostRange{lo, lo + static_cast<unsigned long long>(bytes), name};
}
// Bytes spanned by a bf16 view of `rows` rows.
int64_t view_bytes(int64_t rows, int64_t row_pitch, int64_t heads, int64_t head_pitch, int64_t dim) {
  if (rows <= 0) return 0;
  return 2 * ((rows - 1) * row_pitch + (heads - 1) * head_pitch + dim);
}
void dbg_packed(const kvq_packed* pk) {
  const int64_t rh = static_cast<int64_t>(pk->rows) * pk->heads;
  if (pk->fmt == KVQ_FMT_FP8) {
    dbg_add(pk->codes, rh * pk->dim, "codes");
    dbg_add(pk->rscale, rh * 4, "rscale");
    return;
  }
  dbg_add(pk->codes, rh * (pk->dim / 2), "codes");
  if (pk->fmt == KVQ_FMT_NVFP4_TENSOR) {
    const int64_t nb = pk->kind == KVQ_KIND_KEY ? static_cast<int64_t>((pk->rows + 15) / 16) * pk->heads * pk->dim
                                                : rh * (pk->dim / 16);
    dbg_add(pk->meta0, nb, "bscale");
    dbg_add(pk->rscale, 4, "rscale");
    return;
  }
  if (pk->fmt == KVQ_FMT_NVFP4) {
    dbg_add(pk->meta0, rh * (pk->dim / 16), "bscale");
    dbg_add(pk->rscale, rh * 4, "rscale");
  } else {
    const int G = pk->group_size;
    const int64_t n = pk->kind == KVQ_KIND_KEY
                          ? static_cast<int64_t>((pk->rows + G - 1) / G) * pk->heads * pk->dim
                          : rh * ((pk->dim + G - 1) / G);
    dbg_add(pk->meta0, 2 * n, "min16");
    dbg_add(pk->meta1, 2 * n, "scale16");
  }
}

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};

// Device memory of the current device, else an error status.
kvq_status check_dev(const void* p, const char* what) {
  if (p == nullptr) return fail(KVQ_ERR_INVALID_ARG, "%s is NULL", what);
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // do not leave the error behind for the launch check
    return fail(KVQ_ERR_NOT_DEVICE_PTR, "%s: cudaPointerGetAttributes failed (%s)", what,
                cudaGetErrorString(e));
  }
  if (a.type != cudaMemoryTypeDevice)
    return fail(KVQ_ERR_NOT_DEVICE_PTR, "%s is not device memory (type %d)", what,
                static_cast<int>(a.type));
  int dev = 0;
  cudaGetDevice(&dev);
  if (a.device != dev)
    return fail(KVQ_ERR_NOT_DEVICE_PTR, "%s lives on device %d, current device is %d", what,
                a.device, dev);
  return KVQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A bf16 view: device, 16-byte base, pitches multiple of 8 elements (16 bytes).
// v8 reports whether every 16-element block starts on a 32-byte boundary.
kvq_status check_view(const void* ptr, int64_t row_pitch, int64_t head_pitch, const char* what,
                      bool& v8) {
  kvq_status st = check_dev(ptr, what);
  if (st != KVQ_OK) return st;
  if (row_pitch < 0 || head_pitch < 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: negative pitch", what);
  if (!aligned(ptr, 16) || row_pitch % 8 != 0 || head_pitch % 8 != 0)
    return fail(KVQ_ERR_MISALIGNED,
                "%s: base must be 16-byte aligned and pitches multiples of 8 elements", what);
  v8 = v8 && aligned(ptr, 32) && row_pitch % 16 == 0 && head_pitch % 16 == 0;
#ifdef KVQ_CHECKED
  if (getenv("KVQ_FORCE_V4") != nullptr) v8 = false;
#endif
  return KVQ_OK;
}

kvq_status check_plane(const void* p, const char* what) {
  kvq_status st = check_dev(p, what);
  if (st != KVQ_OK) return st;
  if (!aligned(p, 16)) return fail(KVQ_ERR_MISALIGNED, "%s must be 16-byte aligned", what);
  return KVQ_OK;
}

kvq_status check_head_dim(int32_t H, int32_t D) {
  if (H <= 0) return fail(KVQ_ERR_INVALID_ARG, "heads must be positive (got %d)", H);
  if (D <= 0 || D % 16 != 0)
    return fail(KVQ_ERR_INVALID_ARG, "head_dim must be a positive multiple of 16 (got %d)", D);
  if (D > 512) return fail(KVQ_ERR_UNSUPPORTED, "head_dim above 512 is not supported (got %d)", D);
  return KVQ_OK;
}

// A pool's format and planes (the bscale plane only for NVFP4).
bool pool_fmt_ok(int32_t f) { return f == KVQ_FMT_NVFP4 || f == KVQ_FMT_FP8; }

kvq_status check_pool_fmt(const kvq_pool* pool) {
  if (!pool_fmt_ok(pool->fmt))
    return fail(KVQ_ERR_INVALID_ARG, "pool fmt must be KVQ_FMT_NVFP4 or KVQ_FMT_FP8 (got %d)", pool->fmt);
  if (pool->v_fmt != 0 && !pool_fmt_ok(pool->v_fmt))
    return fail(KVQ_ERR_INVALID_ARG, "pool v_fmt must be 0, KVQ_FMT_NVFP4 or KVQ_FMT_FP8 (got %d)",
                pool->v_fmt);
  return KVQ_OK;
}

// Format of plane j (0 = K, 1 = V).
int32_t plane_fmt(const kvq_pool* pool, int j) {
  return (j == 1 && pool->v_fmt != 0) ? pool->v_fmt : pool->fmt;
}

kvq_status check_pool_plane(int32_t fmt, const kvq_plane* pl) {
  kvq_status st;
  if ((st = check_plane(pl->codes, "pool codes")) != KVQ_OK) return st;
  if (fmt == KVQ_FMT_NVFP4 && (st = check_plane(pl->bscale, "pool bscale")) != KVQ_OK) return st;
  return check_plane(pl->rscale, "pool rscale");
}
int64_t code_bytes_per_row(int32_t fmt, int32_t D) { return fmt == KVQ_FMT_FP8 ? D : D / 2; }

int lanes_for(int32_t D) {
  int nb = D / 16, L = 1;
  while (L < nb) L <<= 1;
  return L;
}

kvq_status launched(cudaError_t e) {
  if (e != cudaSuccess)
    return fail(KVQ_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

bool fits_u31(int64_t v) { return v >= 0 && v < (int64_t{1} << 31); }

kvq_status check_packed(const kvq_packed* pk, const char* what) {
  if (pk == nullptr) return fail(KVQ_ERR_INVALID_ARG, "%s is NULL", what);
  kvq_status st = check_head_dim(pk->heads, pk->dim);
  if (st != KVQ_OK) return st;
  if (pk->rows < 0) return fail(KVQ_ERR_INVALID_ARG, "%s: negative rows", what);
  if (pk->fmt == KVQ_FMT_NVFP4) {
    if (pk->group_size != 16 && pk->group_size != 0)
      return fail(KVQ_ERR_INVALID_ARG, "%s: NVFP4 groups are 16 values", what);
    if (pk->rows == 0) return KVQ_OK;
    if ((st = check_plane(pk->codes, "codes")) != KVQ_OK) return st;
    if ((st = check_plane(pk->meta0, "meta0 (block scales)")) != KVQ_OK) return st;
    if ((st = check_plane(pk->rscale, "rscale")) != KVQ_OK) return st;
  } else if (pk->fmt == KVQ_FMT_FP8) {
    if (pk->rows == 0) return KVQ_OK;
    if ((st = check_plane(pk->codes, "codes")) != KVQ_OK) return st;
    if ((st = check_plane(pk->rscale, "rscale")) != KVQ_OK) return st;
  } else if (pk->fmt == KVQ_FMT_NVFP4_TENSOR) {
    if (pk->group_size != 16 && pk->group_size != 0)
      return fail(KVQ_ERR_INVALID_ARG, "%s: NVFP4 groups are 16 values", what);
    if (pk->kind != KVQ_KIND_KEY && pk->kind != KVQ_KIND_VALUE)
      return fail(KVQ_ERR_INVALID_ARG, "%s: kind must be KEY or VALUE", what);
    if (!fits_u31(static_cast<int64_t>(pk->rows) * pk->heads * pk->dim))
      return fail(KVQ_ERR_UNSUPPORTED, "%s: rows x heads x dim too large", what);
    if (pk->rows == 0) return KVQ_OK;
    if ((st = check_plane(pk->codes, "codes")) != KVQ_OK) return st;
    if ((st = check_plane(pk->meta0, "meta0 (block scales)")) != KVQ_OK) return st;
    if ((st = check_plane(pk->rscale, "rscale")) != KVQ_OK) return st;
  } else if (pk->fmt == KVQ_FMT_INT4) {
    const int G = pk->group_size;
    if (!(G == 16 || G == 32 || G == 64 || G == 128 || G == 256 || G == 512))
      return fail(KVQ_ERR_UNSUPPORTED, "%s: INT4 group size must be 16..512, a power of two (got %d)",
                  what, G);
    if (pk->kind != KVQ_KIND_KEY && pk->kind != KVQ_KIND_VALUE)
      return fail(KVQ_ERR_INVALID_ARG, "%s: kind must be KEY or VALUE", what);
    if (pk->rows == 0) return KVQ_OK;
    if ((st = check_plane(pk->codes, "codes")) != KVQ_OK) return st;
    if ((st = check_plane(pk->meta0, "meta0 (fp16 minimum)")) != KVQ_OK) return st;
    if ((st = check_plane(pk->meta1, "meta1 (fp16 scale)")) != KVQ_OK) return st;
  } else {
    return fail(KVQ_ERR_INVALID_ARG, "%s: unknown format %d", what, pk->fmt);
  }
  if (!fits_u31(static_cast<int64_t>(pk->rows) * pk->heads * 2))
    return fail(KVQ_ERR_UNSUPPORTED, "%s: rows x heads too large", what);
  return KVQ_OK;
}

PayloadRef payload_ref(const kvq_packed* pk) {
  PayloadRef r;
  r.fmt = pk->fmt;
  r.kind = pk->kind;
  r.G = pk->group_size;
  r.codes = pk->codes;
  r.meta0 = pk->meta0;
  r.meta1 = pk->meta1;
  r.rscale = pk->rscale;
  r.rs_stride = 1;
  r.rows = pk->rows;
  return r;
}

}  // namespace

dbg::HostRange* dbg::pending(int* n) {
  *n = g_nranges;
  return g_ranges;
}

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 148;
  if (g_sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 148;
  }
  return g_sms[dev];
}

namespace {
struct OccEntry {
  const void* kernel;
  int threads;
  size_t smem;
  int dev;
  int occ;
};
constexpr int kOccEntries = 512;
OccEntry g_occ[kOccEntries];
int g_nocc = 0;
std::mutex g_occ_mu;
}  // namespace

int cached_occupancy(const void* kernel, int threads, size_t smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_occ_mu);
  for (int i = 0; i < g_nocc; ++i)
    if (g_occ[i].kernel == kernel && g_occ[i].threads == threads && g_occ[i].smem == smem && g_occ[i].dev == dev)
      return g_occ[i].occ;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    occ = 0;
  }
  if (occ < 1) occ = 1;
  if (g_nocc < kOccEntries) g_occ[g_nocc++] = OccEntry{kernel, threads, smem, dev, occ};
  return occ;
}

}  // namespace kvq

using namespace kvq;

namespace {

// Scatter of the given tensors (K and/or V), whose planes share format fmt.
kvq_status scatter_impl(const kvq_bf16_in* k, const kvq_bf16_in* v, int32_t num_tokens,
                        const int64_t* slot_ids, const kvq_pool* pool, int32_t fmt,
                        uint32_t* dev_status, kvq_stream_t stream) {
  kvq_status st;
  const int ntensors = (k != nullptr) + (v != nullptr);
  EncodeParams p{};
  bool v8 = true;
  int i = 0;
  const kvq_bf16_in* src[2] = {k, v};
  const kvq_plane* dst[2] = {&pool->k, &pool->v};
  const char* names[2] = {"k", "v"};
  for (int j = 0; j < 2; ++j) {
    if (src[j] == nullptr) continue;
    if ((st = check_view(src[j]->ptr, src[j]->row_pitch, src[j]->head_pitch, names[j], v8)) != KVQ_OK)
      return st;
    if ((st = check_pool_plane(fmt, dst[j])) != KVQ_OK) return st;
    EncodeTensor& t = p.ten[i++];
    t.x = static_cast<const uint16_t*>(src[j]->ptr);
    t.row_pitch = src[j]->row_pitch;
    t.head_pitch = src[j]->head_pitch;
    t.dst = Nvfp4Planes{dst[j]->codes, dst[j]->bscale, dst[j]->rscale};
  }
  p.ntensors = ntensors;
  p.rows_per_tensor = static_cast<uint32_t>(num_tokens) * static_cast<uint32_t>(pool->num_heads);
  p.div_h = FastDiv(static_cast<uint32_t>(pool->num_heads));
  p.H = pool->num_heads;
  p.nb = pool->head_dim / 16;
  p.slot_ids = slot_ids;
  p.num_slots = pool->num_slots;
  p.status = dev_status;
  dbg_clear();
  for (int j = 0; j < 2; ++j) {
    if (src[j] == nullptr) continue;
    dbg_add(src[j]->ptr, view_bytes(num_tokens, src[j]->row_pitch, pool->num_heads, src[j]->head_pitch, pool->head_dim), names[j]);
    const int64_t rh = pool->num_slots * pool->num_heads;
    dbg_add(dst[j]->codes, rh * code_bytes_per_row(fmt, pool->head_dim), "pool codes");
    if (fmt == KVQ_FMT_NVFP4) dbg_add(dst[j]->bscale, rh * (pool->head_dim / 16), "pool bscale");
    dbg_add(dst[j]->rscale, rh * 4, "pool rscale");
  }
  dbg_add(slot_ids, 8ll * num_tokens, "slot_ids");
  dbg_add(dev_status, 4, "status");
  return launched(launch_nvfp4_encode(p, kEncScatter, fmt, v8, reinterpret_cast<cudaStream_t>(stream)));
}

// Restore of the given tensors (K and/or V), whose planes share format fmt.
kvq_status restore_impl(const kvq_pool* pool, const int32_t* block_table, int32_t num_seqs,
                        int32_t max_blocks, const int32_t* seq_lens, int32_t max_seq_len,
                        const kvq_bf16_out* k_out, const kvq_bf16_out* v_out, int32_t fmt,
                        uint32_t* dev_status, kvq_stream_t stream) {
  kvq_status st;
  const int ntensors = (k_out != nullptr) + (v_out != nullptr);
  DecodeParams p{};
  bool v8 = true;
  int i = 0;
  const kvq_bf16_out* out[2] = {k_out, v_out};
  const kvq_plane* src[2] = {&pool->k, &pool->v};
  const char* names[2] = {"k_out", "v_out"};
  for (int j = 0; j < 2; ++j) {
    if (out[j] == nullptr) continue;
    if ((st = check_view(out[j]->ptr, out[j]->row_pitch, out[j]->head_pitch, names[j], v8)) != KVQ_OK)
      return st;
    if ((st = check_pool_plane(fmt, src[j])) != KVQ_OK) return st;
    DecodeTensor& t = p.ten[i++];
    t.codes = src[j]->codes;
    t.bscale = src[j]->bscale;
    t.rscale = src[j]->rscale;
    t.y = static_cast<uint16_t*>(out[j]->ptr);
    t.row_pitch = out[j]->row_pitch;
    t.head_pitch = out[j]->head_pitch;
  }
  p.ntensors = ntensors;
  p.rows_per_tensor = static_cast<uint32_t>(num_seqs) * static_cast<uint32_t>(max_seq_len) *
                      static_cast<uint32_t>(pool->num_heads);
  p.div_h = FastDiv(static_cast<uint32_t>(pool->num_heads));
  p.div_tmax = FastDiv(static_cast<uint32_t>(max_seq_len));
  p.div_bs = FastDiv(static_cast<uint32_t>(pool->block_size));
  p.H = pool->num_heads;
  p.nb = pool->head_dim / 16;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks;
  p.tmax = max_seq_len;
  const int64_t cap = static_cast<int64_t>(max_blocks) * pool->block_size;
  p.seq_cap = static_cast<int32_t>(cap < max_seq_len ? cap : max_seq_len);
  p.num_blocks = pool->num_slots / pool->block_size;
  p.block_size = pool->block_size;
  p.status = dev_status;
  dbg_clear();
  for (int j = 0; j < 2; ++j) {
    if (out[j] == nullptr) continue;
    dbg_add(out[j]->ptr, view_bytes(static_cast<int64_t>(num_seqs) * max_seq_len, out[j]->row_pitch, pool->num_heads, out[j]->head_pitch, pool->head_dim), names[j]);
    const int64_t rh = pool->num_slots * pool->num_heads;
    dbg_add(src[j]->codes, rh * code_bytes_per_row(fmt, pool->head_dim), "pool codes");
    if (fmt == KVQ_FMT_NVFP4) dbg_add(src[j]->bscale, rh * (pool->head_dim / 16), "pool bscale");
    dbg_add(src[j]->rscale, rh * 4, "pool rscale");
  }
  dbg_add(block_table, 4ll * num_seqs * max_blocks, "block_table");
  dbg_add(seq_lens, 4ll * num_seqs, "seq_lens");
  dbg_add(dev_status, 4, "status");
  return launched(launch_nvfp4_decode(p, kDecRestore, fmt, v8, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

KVQ_API kvq_status kvq_quant_scatter(const kvq_bf16_in* k, const kvq_bf16_in* v,
                                     int32_t num_tokens, const int64_t* slot_ids,
                                     const kvq_pool* pool, uint32_t* dev_status,
                                     kvq_stream_t stream) {
  if (pool == nullptr) return fail(KVQ_ERR_INVALID_ARG, "pool is NULL");
  if (check_pool_fmt(pool) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  if (k == nullptr && v == nullptr) return fail(KVQ_ERR_INVALID_ARG, "both k and v are NULL");
  if (num_tokens < 0) return fail(KVQ_ERR_INVALID_ARG, "negative num_tokens");
  kvq_status st = check_head_dim(pool->num_heads, pool->head_dim);
  if (st != KVQ_OK) return st;
  if (pool->block_size <= 0 || pool->num_slots < 0 || pool->num_slots % pool->block_size != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_slots must be a non-negative multiple of block_size");
  if (num_tokens == 0) return KVQ_OK;
  const int ntensors = (k != nullptr) + (v != nullptr);
  if (!fits_u31(static_cast<int64_t>(num_tokens) * pool->num_heads * ntensors))
    return fail(KVQ_ERR_UNSUPPORTED, "num_tokens x heads too large");
  if ((st = check_dev(slot_ids, "slot_ids")) != KVQ_OK) return st;
  if (dev_status != nullptr && (st = check_dev(dev_status, "dev_status")) != KVQ_OK) return st;
  const int32_t fk = plane_fmt(pool, 0), fv = plane_fmt(pool, 1);
  if (k != nullptr && v != nullptr && fk != fv) {  // split formats: one launch per plane
    if ((st = scatter_impl(k, nullptr, num_tokens, slot_ids, pool, fk, dev_status, stream)) != KVQ_OK)
      return st;
    return scatter_impl(nullptr, v, num_tokens, slot_ids, pool, fv, dev_status, stream);
  }
  return scatter_impl(k, v, num_tokens, slot_ids, pool, k != nullptr ? fk : fv, dev_status, stream);
}

KVQ_API kvq_status kvq_restore(const kvq_pool* pool, const int32_t* block_table,
                               int32_t num_seqs, int32_t max_blocks, const int32_t* seq_lens,
                               int32_t max_seq_len, const kvq_bf16_out* k_out,
                               const kvq_bf16_out* v_out, uint32_t* dev_status,
                               kvq_stream_t stream) {
  if (pool == nullptr) return fail(KVQ_ERR_INVALID_ARG, "pool is NULL");
  if (k_out == nullptr && v_out == nullptr)
    return fail(KVQ_ERR_INVALID_ARG, "both k_out and v_out are NULL");
  if (check_pool_fmt(pool) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  kvq_status st = check_head_dim(pool->num_heads, pool->head_dim);
  if (st != KVQ_OK) return st;
  if (pool->block_size <= 0 || pool->num_slots < 0 || pool->num_slots % pool->block_size != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_slots must be a non-negative multiple of block_size");
  if (num_seqs < 0 || max_blocks < 0 || max_seq_len < 0)
    return fail(KVQ_ERR_INVALID_ARG, "negative num_seqs, max_blocks or max_seq_len");
  if (num_seqs == 0 || max_seq_len == 0) return KVQ_OK;
  const int ntensors = (k_out != nullptr) + (v_out != nullptr);
  if (!fits_u31(static_cast<int64_t>(num_seqs) * max_seq_len * pool->num_heads * ntensors))
    return fail(KVQ_ERR_UNSUPPORTED, "num_seqs x max_seq_len x heads too large");
  if ((st = check_dev(block_table, "block_table")) != KVQ_OK) return st;
  if ((st = check_dev(seq_lens, "seq_lens")) != KVQ_OK) return st;
  if (dev_status != nullptr && (st = check_dev(dev_status, "dev_status")) != KVQ_OK) return st;

  const int32_t fk = plane_fmt(pool, 0), fv = plane_fmt(pool, 1);
  if (k_out != nullptr && v_out != nullptr && fk != fv) {  // split formats: one launch per plane
    if ((st = restore_impl(pool, block_table, num_seqs, max_blocks, seq_lens, max_seq_len, k_out,
                           nullptr, fk, dev_status, stream)) != KVQ_OK)
      return st;
    return restore_impl(pool, block_table, num_seqs, max_blocks, seq_lens, max_seq_len, nullptr, v_out,
                        fv, dev_status, stream);
  }
  return restore_impl(pool, block_table, num_seqs, max_blocks, seq_lens, max_seq_len, k_out, v_out,
                      k_out != nullptr ? fk : fv, dev_status, stream);
}

KVQ_API kvq_status kvq_pack(const kvq_bf16_in* x, const kvq_packed* out, kvq_stream_t stream) {
  kvq_status st = check_packed(out, "out");
  if (st != KVQ_OK) return st;
  if (x == nullptr) return fail(KVQ_ERR_INVALID_ARG, "x is NULL");
  if (out->rows == 0) return KVQ_OK;
  bool v8 = true;
  if ((st = check_view(x->ptr, x->row_pitch, x->head_pitch, "x", v8)) != KVQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dbg_clear();
  dbg_add(x->ptr, view_bytes(out->rows, x->row_pitch, out->heads, x->head_pitch, out->dim), "x");
  dbg_packed(out);
  if (out->fmt == KVQ_FMT_NVFP4_TENSOR) {
    TensorNvfp4Params p{};
    p.x = static_cast<const uint16_t*>(x->ptr);
    p.row_pitch = x->row_pitch;
    p.head_pitch = x->head_pitch;
    p.codes = out->codes;
    p.bscale = static_cast<uint8_t*>(out->meta0);
    p.rscale = out->rscale;
    p.rows = out->rows;
    p.H = out->heads;
    p.D = out->dim;
    p.kind = out->kind;
    p.div_h = FastDiv(static_cast<uint32_t>(out->heads));
    p.div_nb = FastDiv(static_cast<uint32_t>(out->dim / 16));
    p.div_np = FastDiv(static_cast<uint32_t>(out->dim / 2));
    return launched(launch_tensor_nvfp4_pack(p, s));
  }
  if (out->fmt == KVQ_FMT_NVFP4 || out->fmt == KVQ_FMT_FP8) {
    EncodeParams p{};
    p.ten[0].x = static_cast<const uint16_t*>(x->ptr);
    p.ten[0].row_pitch = x->row_pitch;
    p.ten[0].head_pitch = x->head_pitch;
    p.ten[0].dst = Nvfp4Planes{out->codes, static_cast<uint8_t*>(out->meta0), out->rscale};
    p.ntensors = 1;
    p.rows_per_tensor = static_cast<uint32_t>(out->rows) * static_cast<uint32_t>(out->heads);
    p.div_h = FastDiv(static_cast<uint32_t>(out->heads));
    p.H = out->heads;
    p.nb = out->dim / 16;
    return launched(launch_nvfp4_encode(p, kEncPack, out->fmt, v8, s));
  }
  Int4EncodeParams p{};
  p.x = static_cast<const uint16_t*>(x->ptr);
  p.row_pitch = x->row_pitch;
  p.head_pitch = x->head_pitch;
  p.dst = Int4Payload{out->codes, static_cast<uint16_t*>(out->meta0),
                      static_cast<uint16_t*>(out->meta1)};
  p.rows = out->rows;
  p.div_h = FastDiv(static_cast<uint32_t>(out->heads));
  p.H = out->heads;
  p.D = out->dim;
  p.G = out->group_size;
  p.kind = out->kind;
  p.residual = 0;
  p.src_rows = out->rows;
  return launched(launch_int4_encode(p, s));
}

KVQ_API kvq_status kvq_unpack(const kvq_packed* in, const kvq_bf16_out* y, kvq_stream_t stream) {
  kvq_status st = check_packed(in, "in");
  if (st != KVQ_OK) return st;
  if (y == nullptr) return fail(KVQ_ERR_INVALID_ARG, "y is NULL");
  if (in->rows == 0) return KVQ_OK;
  bool v8 = true;
  if ((st = check_view(y->ptr, y->row_pitch, y->head_pitch, "y", v8)) != KVQ_OK) return st;
  if (in->fmt == KVQ_FMT_NVFP4_TENSOR && in->kind == KVQ_KIND_VALUE) {
    // V blocks run along channels: the row codec's layout with one scale shared by
    // every row, decoded by the row-codec decode kernel with a row-scale stride of 0
    UnpackParams u{};
    u.pay = payload_ref(in);
    u.pay.fmt = KVQ_FMT_NVFP4;
    u.pay.rs_stride = 0;
    u.H = in->heads;
    u.D = in->dim;
    u.nb = in->dim / 16;
    u.div_h = FastDiv(static_cast<uint32_t>(in->heads));
    u.total_rows = static_cast<uint32_t>(in->rows) * static_cast<uint32_t>(in->heads);
    u.y = static_cast<uint16_t*>(y->ptr);
    u.y_row_pitch = y->row_pitch;
    u.y_head_pitch = y->head_pitch;
    u.mode = 0;
    dbg_clear();
    dbg_add(y->ptr, view_bytes(in->rows, y->row_pitch, in->heads, y->head_pitch, in->dim), "y");
    dbg_packed(in);
    return launched(launch_payload_decode(u, lanes_for(in->dim), v8, reinterpret_cast<cudaStream_t>(stream)));
  }
  if (in->fmt == KVQ_FMT_NVFP4_TENSOR) {
    TensorNvfp4Params p{};
    p.codes = in->codes;
    p.bscale = static_cast<uint8_t*>(in->meta0);
    p.rscale = in->rscale;
    p.y = static_cast<uint16_t*>(y->ptr);
    p.y_row_pitch = y->row_pitch;
    p.y_head_pitch = y->head_pitch;
    p.rows = in->rows;
    p.H = in->heads;
    p.D = in->dim;
    p.kind = in->kind;
    p.div_h = FastDiv(static_cast<uint32_t>(in->heads));
    p.div_nb = FastDiv(static_cast<uint32_t>(in->dim / 16));
    p.div_np = FastDiv(static_cast<uint32_t>(in->dim / 2));
    dbg_clear();
    dbg_add(y->ptr, view_bytes(in->rows, y->row_pitch, in->heads, y->head_pitch, in->dim), "y");
    dbg_packed(in);
    return launched(launch_tensor_nvfp4_unpack(p, reinterpret_cast<cudaStream_t>(stream)));
  }
  UnpackParams u{};
  u.pay = payload_ref(in);
  u.H = in->heads;
  u.D = in->dim;
  u.nb = in->dim / 16;
  u.div_h = FastDiv(static_cast<uint32_t>(in->heads));
  u.total_rows = static_cast<uint32_t>(in->rows) * static_cast<uint32_t>(in->heads);
  u.y = static_cast<uint16_t*>(y->ptr);
  u.y_row_pitch = y->row_pitch;
  u.y_head_pitch = y->head_pitch;
  u.mode = 0;
  dbg_clear();
  dbg_add(y->ptr, view_bytes(in->rows, y->row_pitch, in->heads, y->head_pitch, in->dim), "y");
  dbg_packed(in);
  return launched(launch_payload_decode(u, lanes_for(in->dim), v8,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

KVQ_API kvq_status kvq_encode_residual(const kvq_bf16_in* cur, const kvq_bf16_in* prev,
                                       int32_t num_rows, const int32_t* pos, int32_t num_pos,
                                       const kvq_packed* payload, int32_t* pos_out,
                                       uint32_t* dev_status, kvq_stream_t stream) {
  kvq_status st = check_packed(payload, "payload");
  if (st == KVQ_OK && payload->fmt == KVQ_FMT_NVFP4_TENSOR)
    return fail(KVQ_ERR_UNSUPPORTED, "residual payloads are NVFP4 rows, FP8 rows or INT4");
  if (st != KVQ_OK) return st;
  if (cur == nullptr || prev == nullptr) return fail(KVQ_ERR_INVALID_ARG, "cur or prev is NULL");
  if (num_rows < 0 || num_pos < 0) return fail(KVQ_ERR_INVALID_ARG, "negative num_rows or num_pos");
  if (pos == nullptr && num_pos != num_rows)
    return fail(KVQ_ERR_INVALID_ARG, "dense residual (pos NULL) needs num_pos == num_rows");
  if (payload->rows != num_pos)
    return fail(KVQ_ERR_INVALID_ARG, "payload rows (%d) must equal num_pos (%d)", payload->rows,
                num_pos);
  if (num_pos == 0) return KVQ_OK;
  bool v8 = true;
  if ((st = check_view(cur->ptr, cur->row_pitch, cur->head_pitch, "cur", v8)) != KVQ_OK) return st;
  if ((st = check_view(prev->ptr, prev->row_pitch, prev->head_pitch, "prev", v8)) != KVQ_OK)
    return st;
  if (pos != nullptr && (st = check_dev(pos, "pos")) != KVQ_OK) return st;
  if (pos_out != nullptr && (st = check_dev(pos_out, "pos_out")) != KVQ_OK) return st;
  if (dev_status != nullptr && (st = check_dev(dev_status, "dev_status")) != KVQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dbg_clear();
  dbg_add(cur->ptr, view_bytes(num_rows, cur->row_pitch, payload->heads, cur->head_pitch, payload->dim), "cur");
  dbg_add(prev->ptr, view_bytes(num_rows, prev->row_pitch, payload->heads, prev->head_pitch, payload->dim), "prev");
  dbg_packed(payload);
  dbg_add(pos, 4ll * num_pos, "pos");
  dbg_add(pos_out, 4ll * num_pos, "pos_out");
  dbg_add(dev_status, 4, "status");
  if (payload->fmt == KVQ_FMT_NVFP4 || payload->fmt == KVQ_FMT_FP8) {
    EncodeParams p{};
    EncodeTensor& t = p.ten[0];
    t.x = static_cast<const uint16_t*>(cur->ptr);
    t.row_pitch = cur->row_pitch;
    t.head_pitch = cur->head_pitch;
    t.prev = static_cast<const uint16_t*>(prev->ptr);
    t.prev_row_pitch = prev->row_pitch;
    t.prev_head_pitch = prev->head_pitch;
    t.dst = Nvfp4Planes{payload->codes, static_cast<uint8_t*>(payload->meta0), payload->rscale};
    p.ntensors = 1;
    p.rows_per_tensor = static_cast<uint32_t>(num_pos) * static_cast<uint32_t>(payload->heads);
    p.div_h = FastDiv(static_cast<uint32_t>(payload->heads));
    p.H = payload->heads;
    p.nb = payload->dim / 16;
    p.pos = pos;
    p.pos_out = pos_out;
    p.src_rows = num_rows;
    p.status = dev_status;
    return launched(launch_nvfp4_encode(p, kEncResidual, payload->fmt, v8, s));
  }
  Int4EncodeParams p{};
  p.x = static_cast<const uint16_t*>(cur->ptr);
  p.row_pitch = cur->row_pitch;
  p.head_pitch = cur->head_pitch;
  p.prev = static_cast<const uint16_t*>(prev->ptr);
  p.prev_row_pitch = prev->row_pitch;
  p.prev_head_pitch = prev->head_pitch;
  p.dst = Int4Payload{payload->codes, static_cast<uint16_t*>(payload->meta0),
                      static_cast<uint16_t*>(payload->meta1)};
  p.rows = num_pos;
  p.div_h = FastDiv(static_cast<uint32_t>(payload->heads));
  p.H = payload->heads;
  p.D = payload->dim;
  p.G = payload->group_size;
  p.kind = payload->kind;
  p.residual = 1;
  p.pos = pos;
  p.pos_out = pos_out;
  p.src_rows = num_rows;
  p.status = dev_status;
  return launched(launch_int4_encode(p, s));
}

KVQ_API kvq_status kvq_decode_residual(const kvq_packed* payload, const int32_t* pos,
                                       int32_t num_pos, const kvq_bf16_in* prev,
                                       int32_t num_rows, const kvq_bf16_out* out,
                                       uint32_t* dev_status, kvq_stream_t stream) {
  kvq_status st = check_packed(payload, "payload");
  if (st == KVQ_OK && payload->fmt == KVQ_FMT_NVFP4_TENSOR)
    return fail(KVQ_ERR_UNSUPPORTED, "residual payloads are NVFP4 rows, FP8 rows or INT4");
  if (st != KVQ_OK) return st;
  if (prev == nullptr || out == nullptr) return fail(KVQ_ERR_INVALID_ARG, "prev or out is NULL");
  if (num_rows < 0 || num_pos < 0) return fail(KVQ_ERR_INVALID_ARG, "negative num_rows or num_pos");
  if (pos == nullptr && num_pos != num_rows)
    return fail(KVQ_ERR_INVALID_ARG, "dense residual (pos NULL) needs num_pos == num_rows");
  if (payload->rows != num_pos)
    return fail(KVQ_ERR_INVALID_ARG, "payload rows (%d) must equal num_pos (%d)", payload->rows,
                num_pos);
  if (!fits_u31(static_cast<int64_t>(num_rows) * payload->heads))
    return fail(KVQ_ERR_UNSUPPORTED, "num_rows x heads too large");
  const bool in_place = out->ptr == prev->ptr && out->row_pitch == prev->row_pitch &&
                        out->head_pitch == prev->head_pitch;
  if (num_rows == 0 || (in_place && num_pos == 0)) return KVQ_OK;
  bool v8 = true;
  if ((st = check_view(prev->ptr, prev->row_pitch, prev->head_pitch, "prev", v8)) != KVQ_OK)
    return st;
  if ((st = check_view(out->ptr, out->row_pitch, out->head_pitch, "out", v8)) != KVQ_OK) return st;
  if (!in_place) {
    // the two views must not share memory
    const int64_t span = 2 * ((static_cast<int64_t>(num_rows) - 1) * prev->row_pitch +
                              (static_cast<int64_t>(payload->heads) - 1) * prev->head_pitch +
                              payload->dim);
    const int64_t ospan = 2 * ((static_cast<int64_t>(num_rows) - 1) * out->row_pitch +
                               (static_cast<int64_t>(payload->heads) - 1) * out->head_pitch +
                               payload->dim);
    const char* a = static_cast<const char*>(prev->ptr);
    const char* b = static_cast<const char*>(out->ptr);
    if (a < b + ospan && b < a + span)
      return fail(KVQ_ERR_INVALID_ARG, "out overlaps prev without being the same view");
  }
  if (pos != nullptr && num_pos > 0 && (st = check_dev(pos, "pos")) != KVQ_OK) return st;
  if (dev_status != nullptr && (st = check_dev(dev_status, "dev_status")) != KVQ_OK) return st;
  UnpackParams u{};
  u.pay = payload_ref(payload);
  u.H = payload->heads;
  u.D = payload->dim;
  u.nb = payload->dim / 16;
  u.div_h = FastDiv(static_cast<uint32_t>(payload->heads));
  u.y = static_cast<uint16_t*>(out->ptr);
  u.y_row_pitch = out->row_pitch;
  u.y_head_pitch = out->head_pitch;
  u.prev = static_cast<const uint16_t*>(prev->ptr);
  u.prev_row_pitch = prev->row_pitch;
  u.prev_head_pitch = prev->head_pitch;
  u.pos = pos;  // non-NULL with num_pos == 0: every row is absent (never dereferenced)
  u.num_pos = num_pos;
  u.src_rows = num_rows;
  u.status = dev_status;
  dbg_clear();
  dbg_add(prev->ptr, view_bytes(num_rows, prev->row_pitch, payload->heads, prev->head_pitch, payload->dim), "prev");
  if (!in_place)
    dbg_add(out->ptr, view_bytes(num_rows, out->row_pitch, payload->heads, out->head_pitch, payload->dim), "out");
  dbg_packed(payload);
  if (num_pos > 0) dbg_add(pos, 4ll * num_pos, "pos");
  dbg_add(dev_status, 4, "status");
  if (in_place) {
    u.mode = 1;
    u.total_rows = static_cast<uint32_t>(num_pos) * static_cast<uint32_t>(payload->heads);
  } else {
    u.mode = 2;
    u.total_rows = static_cast<uint32_t>(num_rows) * static_cast<uint32_t>(payload->heads);
  }
  return launched(launch_payload_decode(u, lanes_for(payload->dim), v8,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

// Splits and tokens per split of a decode-attention call (tokens per split a multiple
// of 64: whole 16-token tiles for each of the 4 warps).
KVQ_API size_t kvq_decode_attention_workspace(int32_t num_seqs, int32_t num_heads, int32_t num_q_heads,
                                              int32_t head_dim, int32_t max_seq_len) {
  return attn_workspace_bytes(num_seqs, num_heads, num_q_heads, head_dim, max_seq_len);
}

}  // extern "C"

namespace {

// Decode attention behind both entry points: the same argument checks, then the split
// partials go to the caller's workspace, or (builtin) to the library's own scratch.
kvq_status decode_attention_impl(const kvq_pool* pool, const int32_t* block_table, int32_t num_seqs,
                                 int32_t max_blocks, const int32_t* seq_lens, int32_t max_seq_len,
                                 const kvq_bf16_in* q, int32_t num_q_heads, float scale,
                                 const kvq_bf16_out* out, void* workspace, size_t workspace_bytes,
                                 bool builtin, uint32_t* dev_status, kvq_stream_t stream) {
  if (pool == nullptr || q == nullptr || out == nullptr)
    return fail(KVQ_ERR_INVALID_ARG, "pool, q and out must not be NULL");
  if (check_pool_fmt(pool) != KVQ_OK) return KVQ_ERR_INVALID_ARG;
  kvq_status st = check_head_dim(pool->num_heads, pool->head_dim);
  if (st != KVQ_OK) return st;
  const int32_t D = pool->head_dim, H = pool->num_heads;
  if (D != 64 && D != 128 && D != 256)
    return fail(KVQ_ERR_UNSUPPORTED, "decode attention supports head_dim 64, 128 or 256 (got %d)", D);
  if (pool->block_size <= 0 || pool->num_slots < 0 || pool->num_slots % pool->block_size != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_slots must be a non-negative multiple of block_size");
  if (num_seqs < 0 || max_blocks < 0 || max_seq_len < 0)
    return fail(KVQ_ERR_INVALID_ARG, "negative num_seqs, max_blocks or max_seq_len");
  if (num_q_heads <= 0 || num_q_heads % H != 0)
    return fail(KVQ_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_heads");
  if (num_q_heads / H > 16) return fail(KVQ_ERR_UNSUPPORTED, "at most 16 query heads per KV head");
  if (!(scale > 0.0f && scale <= 3.4028235e38f))
    return fail(KVQ_ERR_INVALID_ARG, "scale must be positive and finite (got %g)", static_cast<double>(scale));
  if (num_seqs > 65535 || H > 65535) return fail(KVQ_ERR_UNSUPPORTED, "num_seqs and num_heads must be <= 65535");
  if (num_seqs == 0) return KVQ_OK;
  if (!fits_u31(static_cast<int64_t>(num_seqs) * num_q_heads * D))
    return fail(KVQ_ERR_UNSUPPORTED, "num_seqs x num_q_heads x head_dim too large");
  bool v8 = true;
  if ((st = check_view(q->ptr, q->row_pitch, q->head_pitch, "q", v8)) != KVQ_OK) return st;
  if ((st = check_view(out->ptr, out->row_pitch, out->head_pitch, "out", v8)) != KVQ_OK) return st;
  const int32_t fk = plane_fmt(pool, 0), fv = plane_fmt(pool, 1);
  if ((st = check_pool_plane(fk, &pool->k)) != KVQ_OK) return st;
  if ((st = check_pool_plane(fv, &pool->v)) != KVQ_OK) return st;
  if ((st = check_dev(block_table, "block_table")) != KVQ_OK) return st;
  if ((st = check_dev(seq_lens, "seq_lens")) != KVQ_OK) return st;
  if (dev_status != nullptr && (st = check_dev(dev_status, "dev_status")) != KVQ_OK) return st;

  AttnParams p{};
  p.max_len = max_seq_len;
  const size_t need = kvq_decode_attention_workspace(num_seqs, H, num_q_heads, D, max_seq_len);
  if (builtin && need > 0) {
    if (need > attn_builtin_scratch_bytes())
      return fail(KVQ_ERR_UNSUPPORTED, "split partials need %zu bytes, more than the built-in %zu", need,
                  attn_builtin_scratch_bytes());
    const cudaError_t e = attn_builtin_scratch(&workspace, &workspace_bytes);
    if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "built-in scratch: %s", cudaGetErrorString(e));
  } else if (need > 0) {
    if ((st = check_dev(workspace, "workspace")) != KVQ_OK) return st;
    if (!aligned(workspace, 16)) return fail(KVQ_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    if (workspace_bytes < need)
      return fail(KVQ_ERR_INVALID_ARG, "workspace too small: %zu bytes, need %zu", workspace_bytes, need);
  }
  p.k = AttnPlane{pool->k.codes, pool->k.bscale, pool->k.rscale};
  p.v = AttnPlane{pool->v.codes, pool->v.bscale, pool->v.rscale};
  p.fmt_k = fk;
  p.fmt_v = fv;
  p.q = static_cast<const uint16_t*>(q->ptr);
  p.q_row_pitch = q->row_pitch;
  p.q_head_pitch = q->head_pitch;
  p.out = static_cast<uint16_t*>(out->ptr);
  p.o_row_pitch = out->row_pitch;
  p.o_head_pitch = out->head_pitch;
  p.ws = static_cast<float*>(workspace);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks;
  const int64_t cap = static_cast<int64_t>(max_blocks) * pool->block_size;
  p.seq_cap = static_cast<int32_t>(cap < max_seq_len ? cap : max_seq_len);
  p.block_size = pool->block_size;
  p.div_bs = FastDiv(static_cast<uint32_t>(pool->block_size));
  p.num_blocks = pool->num_slots / pool->block_size;
  p.S = num_seqs;
  p.H = H;
  p.Hq = num_q_heads;
  p.D = D;
  p.group = num_q_heads / H;
  p.scale = scale;
  p.status = dev_status;
  dbg_clear();
  const int64_t rh = pool->num_slots * H;
  dbg_add(pool->k.codes, rh * code_bytes_per_row(fk, D), "k codes");
  if (fk == KVQ_FMT_NVFP4) dbg_add(pool->k.bscale, rh * (D / 16), "k bscale");
  dbg_add(pool->k.rscale, rh * 4, "k rscale");
  dbg_add(pool->v.codes, rh * code_bytes_per_row(fv, D), "v codes");
  if (fv == KVQ_FMT_NVFP4) dbg_add(pool->v.bscale, rh * (D / 16), "v bscale");
  dbg_add(pool->v.rscale, rh * 4, "v rscale");
  dbg_add(q->ptr, view_bytes(num_seqs, q->row_pitch, num_q_heads, q->head_pitch, D), "q");
  dbg_add(out->ptr, view_bytes(num_seqs, out->row_pitch, num_q_heads, out->head_pitch, D), "out");
  dbg_add(block_table, 4ll * num_seqs * max_blocks, "block_table");
  dbg_add(seq_lens, 4ll * num_seqs, "seq_lens");
  if (need > 0) dbg_add(workspace, static_cast<int64_t>(need), "workspace");
  dbg_add(dev_status, 4, "status");
  return launched(launch_decode_attention(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

KVQ_API kvq_status kvq_decode_attention(const kvq_pool* pool, const int32_t* block_table,
                                        int32_t num_seqs, int32_t max_blocks, const int32_t* seq_lens,
                                        int32_t max_seq_len, const kvq_bf16_in* q, int32_t num_q_heads,
                                        float scale, const kvq_bf16_out* out, void* workspace,
                                        size_t workspace_bytes, uint32_t* dev_status,
                                        kvq_stream_t stream) {
  return decode_attention_impl(pool, block_table, num_seqs, max_blocks, seq_lens, max_seq_len, q, num_q_heads,
                               scale, out, workspace, workspace_bytes, false, dev_status, stream);
}

KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_pool* pool, const int32_t* block_table,
                                                int32_t num_seqs, int32_t max_blocks,
                                                const int32_t* seq_lens, int32_t max_seq_len,
                                                const kvq_bf16_in* q, int32_t num_q_heads, float scale,
                                                const kvq_bf16_out* out, uint32_t* dev_status,
                                                kvq_stream_t stream) {
  return decode_attention_impl(pool, block_table, num_seqs, max_blocks, seq_lens, max_seq_len, q, num_q_heads,
                               scale, out, nullptr, 0, true, dev_status, stream);
}

KVQ_API size_t kvq_storage_bytes(kvq_format fmt, kvq_kind kind, int32_t group_size, int64_t rows,
                                 int32_t heads, int32_t dim) {
  if (rows < 0 || heads <= 0 || dim <= 0) return 0;
  const int64_t rh = rows * heads;
  if (fmt == KVQ_FMT_NVFP4) {
    if (dim % 16 != 0) return 0;
    return static_cast<size_t>(rh * (dim / 2 + dim / 16 + 4));
  }
  if (fmt == KVQ_FMT_FP8) return static_cast<size_t>(rh * (dim + 4));
  if (fmt == KVQ_FMT_NVFP4_TENSOR) {
    if (dim % 16 != 0 || (kind != KVQ_KIND_KEY && kind != KVQ_KIND_VALUE)) return 0;
    const int64_t blocks = kind == KVQ_KIND_KEY ? ((rows + 15) / 16) * heads * dim : rh * (dim / 16);
    return static_cast<size_t>(rh * (dim / 2) + blocks + 4);
  }
  if (fmt == KVQ_FMT_INT4) {
    if (dim % 2 != 0 || group_size <= 0) return 0;
    const int64_t codes = rh * (dim / 2);
    int64_t groups;
    if (kind == KVQ_KIND_KEY)
      groups = ((rows + group_size - 1) / group_size) * heads * dim;
    else if (kind == KVQ_KIND_VALUE)
      groups = rh * ((dim + group_size - 1) / group_size);
    else
      return 0;
    return static_cast<size_t>(codes + groups * 4);
  }
  return 0;
}

KVQ_API const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_MISALIGNED: return "KVQ_ERR_MISALIGNED";
    case KVQ_ERR_NOT_DEVICE_PTR: return "KVQ_ERR_NOT_DEVICE_PTR";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
  }
  return "KVQ_ERR_UNKNOWN";
}

KVQ_API const char* kvq_last_error(void) { return g_last_error; }

}  // extern "C"
