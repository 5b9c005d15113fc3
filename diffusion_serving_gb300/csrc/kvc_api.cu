// C-ABI entry points of libkvc.so (declared and documented in include/kvc.h):
// host-side validation, handle state and kernel selection.  Every call only
// enqueues work on the caller's stream; nothing here allocates device memory.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "kvc_internal.h"

namespace {

// Blocks the split-KV decode kernel aims for (one per SM of a 152-SM GB300).
// A constant, so that workspace sizes do not depend on the device queried.
constexpr int kDecodeTargetBlocks = 152;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int elem_bytes(int dtype) { return dtype == KVC_F32 ? 4 : 2; }

// Validate a config; on success store the per-row slot count in *cap.
int check_cfg(const kvc_config* cfg, int* cap) {
  if (cfg == nullptr) return KVC_ERR_ARG;
  if (cfg->batch < 1 || cfg->heads < 1 || cfg->kv_heads < 1 || cfg->heads % cfg->kv_heads) return KVC_ERR_ARG;
  if (cfg->dtype < KVC_F32 || cfg->dtype > KVC_BF16) return KVC_ERR_ARG;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (!(cfg->softmax_scale >= 0.f) || isinf(cfg->softmax_scale)) return KVC_ERR_ARG;
  switch (cfg->layout) {
    case KVC_CIRCULAR:
      if (cfg->chunk < 1 || cfg->sink < 0 || cfg->window <= cfg->sink) return KVC_ERR_ARG;
      if (cfg->sink % cfg->chunk || (cfg->window - cfg->sink) % cfg->chunk) return KVC_ERR_ARG;
      *cap = cfg->window;
      break;
    case KVC_LINEAR:
    case KVC_PACKED:
      if (cfg->capacity < 1) return KVC_ERR_ARG;
      *cap = cfg->capacity;
      break;
    default:
      return KVC_ERR_ARG;
  }
  // element offsets of the store must fit the kernels' 64-bit arithmetic; row counts
  // must fit int32
  const int64_t rows = (int64_t)(cfg->layout == KVC_PACKED ? 1 : cfg->batch) * (*cap);
  if (rows > INT32_MAX) return KVC_ERR_ARG;
  return KVC_OK;
}

int decode_splits(const kvc_config& cfg, int cap) {
  const int pairs = cfg.batch * cfg.kv_heads;
  int n = (kDecodeTargetBlocks + pairs - 1) / pairs;
  if (n > KVC_DECODE_MAX_SPLITS) n = KVC_DECODE_MAX_SPLITS;
  if (n > cap) n = cap;
  return n < 1 ? 1 : n;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int launched(cudaError_t e) { return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA; }

// The write kernels count the K and V source rows of a call (2 x B x n_tokens) in int32.
bool write_rows_overflow(const kvc_cache* c, int32_t n_tokens) {
  return 2LL * c->cfg.batch * n_tokens > INT32_MAX;
}

constexpr uint32_t kFlags = KVC_CAUSAL | KVC_KERNEL_SIMT | KVC_DETERMINISTIC;   // every attend flag

// Kernel choice by shape only: fp32 (or the SIMT flag) -> fp32-FMA kernel; one query
// token -> split-KV decode; bf16/fp16 with D = 128 -> tensor-core kernel; otherwise the
// fp32-FMA kernel.
int attend_impl(kvc_cache* c, const void* q, void* out, float* lse, int n_q, uint32_t flags, cudaStream_t s) {
  const bool causal = (flags & KVC_CAUSAL) != 0;
  if ((flags & KVC_KERNEL_SIMT) || c->cfg.dtype == KVC_F32)
    return launched(kvc_launch_attn_simt(c, q, out, n_q, causal, lse, s));
  if (n_q == 1 && c->dec_splits > 0)
    return launched(kvc_launch_decode(c, q, out, lse, (flags & KVC_DETERMINISTIC) != 0, s));
  if (c->tc_ok) return launched(kvc_launch_attn_tc(c, q, out, n_q, causal, lse, s));
  return launched(kvc_launch_attn_simt(c, q, out, n_q, causal, lse, s));
}

}  // namespace

// ---- TMA descriptors ---------------------------------------------------------
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}
}  // namespace

bool kvc_make_tile_map(CUtensorMap* m, int dtype, const void* base, int D, uint64_t d1, uint64_t d2, uint64_t d3,
                       uint32_t box_rows, kvc_box box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr || (dtype != KVC_BF16 && dtype != KVC_F16)) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, d1, d2, d3};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2ull, d1 * D * 2ull, d2 * d1 * D * 2ull};
  const cuuint32_t inner = box == KVC_BOX_SW64 ? 32u : 64u;
  const cuuint32_t boxdim[4] = {inner, 1, box_rows, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t = dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw = box == KVC_BOX_SW64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(m, t, 4, const_cast<void*>(base), dims, strides, boxdim, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int kvc_internal_check_config(const kvc_config* cfg, int* cap) { return check_cfg(cfg, cap); }
int kvc_internal_decode_splits(const kvc_config& cfg, int cap) { return decode_splits(cfg, cap); }

extern "C" {

size_t kvc_meta_bytes(const kvc_config* cfg) {
  int cap = 0;
  if (check_cfg(cfg, &cap) != KVC_OK) return 0;
  const size_t words = (size_t)kvc_meta_cu(cfg->batch) + cfg->batch + 1;
  return (words * 4 + 255) & ~(size_t)255;
}

size_t kvc_workspace_bytes(const kvc_config* cfg) {
  int cap = 0;
  if (check_cfg(cfg, &cap) != KVC_OK) return 0;
  if (!kvc_decode_supported(*cfg)) return 0;
  const size_t b = kvc_decode_workspace_bytes(*cfg, decode_splits(*cfg, cap));
  return (b + 255) & ~(size_t)255;
}

int kvc_create(const kvc_config* cfg, void* k_store, void* v_store, void* meta, void* workspace, void* stream,
               kvc_cache** out) {
  int cap = 0;
  if (out == nullptr) return KVC_ERR_ARG;
  *out = nullptr;
  int rc = check_cfg(cfg, &cap);
  if (rc != KVC_OK) return rc;
  if (!k_store || !v_store || !meta || !aligned16(k_store) || !aligned16(v_store) || !aligned16(meta))
    return KVC_ERR_ARG;
  const size_t ws_bytes = kvc_workspace_bytes(cfg);
  if (ws_bytes > 0 && (workspace == nullptr || !aligned16(workspace))) return KVC_ERR_ARG;

  kvc_cache* c = new (std::nothrow) kvc_cache();
  if (c == nullptr) return KVC_ERR_ARG;
  c->cfg = *cfg;
  c->cap = cap;
  c->eb = elem_bytes(cfg->dtype);
  c->scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0f / sqrtf((float)cfg->head_dim);
  c->k = k_store;
  c->v = v_store;
  c->meta = reinterpret_cast<int32_t*>(meta);
  c->lens = c->meta;
  c->bound = nullptr;
  c->ws = workspace;
  c->dec_splits = kvc_decode_supported(*cfg) ? decode_splits(*cfg, cap) : 0;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return KVC_ERR_CUDA;
  }
  if (c->dec_splits > 0 && (!kvc_make_decode_maps(c) || kvc_prepare_decode(c) != cudaSuccess)) {
    delete c;
    return KVC_ERR_CUDA;
  }
  c->tc_ok = kvc_tc_supported(*cfg) && kvc_tc_make_kv_maps(c);
  cudaStream_t s = as_stream(stream);
  if (cudaMemsetAsync(meta, 0, kvc_meta_bytes(cfg), s) != cudaSuccess ||
      (ws_bytes > 0 && cudaMemsetAsync(workspace, 0, ws_bytes, s) != cudaSuccess)) {
    delete c;
    return KVC_ERR_CUDA;
  }
  *out = c;
  return KVC_OK;
}

int kvc_advance(kvc_cache* c, int32_t row, int32_t n_tokens, void* stream) {
  if (c == nullptr || row >= c->cfg.batch) return KVC_ERR_ARG;
  switch (c->cfg.layout) {
    case KVC_CIRCULAR:
      if (n_tokens != c->cfg.chunk) return KVC_ERR_ARG;
      break;
    case KVC_LINEAR:
      if (n_tokens < 1) return KVC_ERR_ARG;
      if (n_tokens > c->cap) return KVC_ERR_RANGE;
      break;
    default:
      return KVC_ERR_UNSUPPORTED;
  }
  return launched(kvc_launch_advance(c, row < 0 ? -1 : row, n_tokens, as_stream(stream)));
}

int kvc_write(kvc_cache* c, const void* k, const void* v, int32_t n_tokens, const int32_t* d_slots, void* stream) {
  if (c == nullptr || !k || !v || !aligned16(k) || !aligned16(v) || n_tokens < 1) return KVC_ERR_ARG;
  // a packed write reads a padded source: rows past each row's length are skipped
  if (n_tokens > c->cap && c->cfg.layout != KVC_PACKED) return KVC_ERR_RANGE;
  if (write_rows_overflow(c, n_tokens)) return KVC_ERR_RANGE;
  if (d_slots != nullptr) {
    if (c->cfg.layout == KVC_PACKED) return KVC_ERR_UNSUPPORTED;
    if (((uintptr_t)d_slots & 3u) != 0) return KVC_ERR_ARG;
  } else if (c->cfg.layout == KVC_CIRCULAR && n_tokens != c->cfg.chunk) {
    return KVC_ERR_ARG;
  }
  return launched(kvc_launch_write(c, k, v, n_tokens, d_slots, as_stream(stream)));
}

int kvc_append(kvc_cache* c, const void* k, const void* v, int32_t n_tokens, void* stream) {
  if (c == nullptr || !k || !v || !aligned16(k) || !aligned16(v) || n_tokens < 1) return KVC_ERR_ARG;
  if (c->cfg.layout != KVC_LINEAR) return KVC_ERR_UNSUPPORTED;
  if (n_tokens > c->cap || write_rows_overflow(c, n_tokens)) return KVC_ERR_RANGE;
  cudaStream_t s = as_stream(stream);
  if (kvc_append_fits(c, n_tokens)) return launched(kvc_launch_append(c, k, v, n_tokens, s));
  const cudaError_t e = kvc_launch_advance(c, -1, n_tokens, s);
  if (e != cudaSuccess) return KVC_ERR_CUDA;
  return launched(kvc_launch_write(c, k, v, n_tokens, nullptr, s));
}

int kvc_append_attend_decode(kvc_cache* c, const void* k_new, const void* v_new, const void* q, void* out,
                             void* stream) {
  if (c == nullptr || !k_new || !v_new || !q || !out) return KVC_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(out)) return KVC_ERR_ARG;
  if (c->cfg.layout != KVC_LINEAR || c->dec_splits <= 0 || c->bound != nullptr) return KVC_ERR_UNSUPPORTED;
  return launched(kvc_launch_decode_append(c, k_new, v_new, q, out, as_stream(stream)));
}

int kvc_write_rope(kvc_cache* c, const void* k, const void* v, int32_t n_tokens, const int32_t* d_slots,
                   const float* d_rope, int32_t rope_positions, void* stream) {
  if (c == nullptr || !k || !v || !aligned16(k) || !aligned16(v) || n_tokens < 1) return KVC_ERR_ARG;
  if (d_rope == nullptr || ((uintptr_t)d_rope & 7u) != 0 || rope_positions < 1) return KVC_ERR_ARG;
  if (n_tokens > c->cap && c->cfg.layout != KVC_PACKED) return KVC_ERR_RANGE;
  if (write_rows_overflow(c, n_tokens)) return KVC_ERR_RANGE;
  if (d_slots != nullptr) {
    if (c->cfg.layout == KVC_PACKED) return KVC_ERR_UNSUPPORTED;
    if (((uintptr_t)d_slots & 3u) != 0) return KVC_ERR_ARG;
  } else if (c->cfg.layout == KVC_CIRCULAR && n_tokens != c->cfg.chunk) {
    return KVC_ERR_ARG;
  }
  return launched(kvc_launch_write_rope(c, k, v, n_tokens, d_slots, d_rope, rope_positions, as_stream(stream)));
}

int kvc_set_lengths(kvc_cache* c, const int32_t* d_kv_len, const int32_t* d_cu_seqlens, void* stream) {
  if (c == nullptr || (d_kv_len == nullptr && d_cu_seqlens == nullptr)) return KVC_ERR_ARG;
  if (d_kv_len != nullptr && c->cfg.layout == KVC_PACKED) return KVC_ERR_UNSUPPORTED;
  if (d_cu_seqlens != nullptr && c->cfg.layout != KVC_PACKED) return KVC_ERR_UNSUPPORTED;
  return launched(kvc_launch_set_lengths(c, d_kv_len, d_cu_seqlens, as_stream(stream)));
}

size_t kvc_lengths_bytes(int32_t batch) {
  if (batch < 1) return 0;
  const size_t words = (size_t)kvc_meta_cu(batch) + batch + 1;
  return (words * 4 + 255) & ~(size_t)255;
}

int kvc_lengths_create(int32_t batch, int32_t layout, int32_t capacity, void* d_block, void* stream,
                       kvc_lengths** out) {
  if (out == nullptr) return KVC_ERR_ARG;
  *out = nullptr;
  if (batch < 1 || capacity < 1 || d_block == nullptr || !aligned16(d_block)) return KVC_ERR_ARG;
  if (layout != KVC_LINEAR && layout != KVC_PACKED) return KVC_ERR_UNSUPPORTED;
  kvc_lengths* L = new (std::nothrow) kvc_lengths();
  if (L == nullptr) return KVC_ERR_ARG;
  L->batch = batch;
  L->layout = layout;
  L->cap = capacity;
  L->block = reinterpret_cast<int32_t*>(d_block);
  if (cudaMemsetAsync(d_block, 0, kvc_lengths_bytes(batch), as_stream(stream)) != cudaSuccess) {
    delete L;
    return KVC_ERR_CUDA;
  }
  *out = L;
  return KVC_OK;
}

int kvc_lengths_set(kvc_lengths* L, const int32_t* d_kv_len, const int32_t* d_cu_seqlens, void* stream) {
  if (L == nullptr || (d_kv_len == nullptr && d_cu_seqlens == nullptr)) return KVC_ERR_ARG;
  if (d_kv_len != nullptr && L->layout == KVC_PACKED) return KVC_ERR_UNSUPPORTED;
  if (d_cu_seqlens != nullptr && L->layout != KVC_PACKED) return KVC_ERR_UNSUPPORTED;
  return launched(kvc_launch_set_lengths_block(L->block, L->batch, L->cap, d_kv_len, d_cu_seqlens,
                                               as_stream(stream)));
}

int kvc_use_lengths(kvc_cache* c, const kvc_lengths* L) {
  if (c == nullptr) return KVC_ERR_ARG;
  if (L == nullptr) {
    c->lens = c->meta;
    c->bound = nullptr;
    return KVC_OK;
  }
  if (L->batch != c->cfg.batch || L->cap > c->cap) return KVC_ERR_ARG;
  if (L->layout != c->cfg.layout) return KVC_ERR_UNSUPPORTED;
  c->lens = L->block;
  c->bound = L;
  return KVC_OK;
}

int kvc_lengths_destroy(kvc_lengths* L) {
  delete L;
  return KVC_OK;
}

int kvc_attend(kvc_cache* c, const void* q, void* out, int32_t n_q, uint32_t flags, void* stream) {
  if (c == nullptr || !q || !out || !aligned16(q) || !aligned16(out) || n_q < 1) return KVC_ERR_ARG;
  if (flags & ~kFlags) return KVC_ERR_ARG;
  if ((flags & KVC_CAUSAL) && c->cfg.layout != KVC_LINEAR) return KVC_ERR_UNSUPPORTED;
  return attend_impl(c, q, out, nullptr, n_q, flags, as_stream(stream));
}

int kvc_attend_lse(kvc_cache* c, const void* q, void* out, float* d_lse, int32_t n_q, uint32_t flags,
                   void* stream) {
  if (c == nullptr || !q || !out || !d_lse || !aligned16(q) || !aligned16(out) || n_q < 1) return KVC_ERR_ARG;
  if (((uintptr_t)d_lse & 3u) != 0 || (flags & ~kFlags)) return KVC_ERR_ARG;
  if ((flags & KVC_CAUSAL) && c->cfg.layout != KVC_LINEAR) return KVC_ERR_UNSUPPORTED;
  return attend_impl(c, q, out, d_lse, n_q, flags, as_stream(stream));
}

int kvc_merge(int32_t dtype, int32_t n_rows, int32_t head_dim, const void* o_a, const float* lse_a, const void* o_b,
              const float* lse_b, void* out, float* lse_out, void* stream) {
  if (dtype < KVC_F32 || dtype > KVC_BF16 || n_rows < 1 || head_dim < 1) return KVC_ERR_ARG;
  if (!o_a || !o_b || !out || !lse_a || !lse_b) return KVC_ERR_ARG;
  return launched(kvc_launch_merge(dtype, n_rows, head_dim, o_a, lse_a, o_b, lse_b, out, lse_out, as_stream(stream)));
}

size_t kvc_roll_scratch_bytes(const kvc_config* cfg) {
  int cap = 0;
  if (check_cfg(cfg, &cap) != KVC_OK || cfg->layout != KVC_CIRCULAR) return 0;
  const int64_t count = cfg->window - cfg->sink - cfg->chunk;
  if (count <= 0) return 0;
  return (size_t)2 * cfg->batch * count * cfg->kv_heads * cfg->head_dim * elem_bytes(cfg->dtype);
}

int kvc_roll_window(kvc_cache* c, void* d_scratch, void* stream) {
  if (c == nullptr) return KVC_ERR_ARG;
  if (c->cfg.layout != KVC_CIRCULAR) return KVC_ERR_UNSUPPORTED;
  if (kvc_roll_scratch_bytes(&c->cfg) > 0 && (d_scratch == nullptr || !aligned16(d_scratch))) return KVC_ERR_ARG;
  return launched(kvc_launch_roll(c, d_scratch, as_stream(stream)));
}

int kvc_reset(kvc_cache* c, int32_t row, void* stream) {
  if (c == nullptr || row >= c->cfg.batch) return KVC_ERR_ARG;
  return launched(kvc_launch_reset(c, row < 0 ? -1 : row, as_stream(stream)));
}

int kvc_get_error(kvc_cache* c, void* stream, int32_t* bits) {
  if (c == nullptr) return KVC_ERR_ARG;
  cudaStream_t s = as_stream(stream);
  int32_t word = 0, shared = 0;
  int32_t* shared_word = c->bound != nullptr ? c->bound->block + KVC_META_ERR : nullptr;
  if (cudaMemcpyAsync(&word, c->meta + KVC_META_ERR, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      (shared_word != nullptr &&
       cudaMemcpyAsync(&shared, shared_word, sizeof(shared), cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (shared != 0 && cudaMemsetAsync(shared_word, 0, sizeof(int32_t), s) != cudaSuccess) return KVC_ERR_CUDA;
  word |= shared;
  if (bits != nullptr) *bits = word;
  if (word == 0) return KVC_OK;
  if (cudaMemsetAsync(c->meta + KVC_META_ERR, 0, sizeof(int32_t), s) != cudaSuccess) return KVC_ERR_CUDA;
  if ((word & KVC_DEV_TIMEOUT) && c->ws != nullptr && c->dec_splits > 0) {
    // a decode kernel that gave up may have left its ticket and tile-claim counters
    // (the last 8 bytes per (row, kv head) of the workspace) off zero
    const size_t raw = kvc_decode_workspace_bytes(c->cfg, c->dec_splits);
    const size_t counters = (size_t)c->cfg.batch * c->cfg.kv_heads * 8;
    if (cudaMemsetAsync(static_cast<unsigned char*>(c->ws) + (raw - counters), 0, counters, s) != cudaSuccess)
      return KVC_ERR_CUDA;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_ERR_DEVICE;
}

int kvc_debug_stall_waits(kvc_cache* c, uint64_t ns) {
  if (c == nullptr) return KVC_ERR_ARG;
  c->debug_stall_ns = ns;
  return KVC_OK;
}

int kvc_destroy(kvc_cache* c) {
  delete c;
  return KVC_OK;
}

const char* kvc_strerror(int code) {
  switch (code) {
    case KVC_OK: return "ok";
    case KVC_ERR_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported configuration or request";
    case KVC_ERR_RANGE: return "length out of range";
    case KVC_ERR_CUDA: return "CUDA error";
    case KVC_ERR_DEVICE: return "device-side error reported";
    default: return "unknown error code";
  }
}

}  // extern "C"
