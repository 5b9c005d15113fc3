// Internal declarations shared by the kvc host layer and its kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

// ---- meta block layout (int32 words; documented in kvc.h) -------------------
#define KVC_META_ERR 0
#define KVC_META_ARRIVE 1   // blocks of an append-then-attend decode launch that have read their lengths
#define KVC_META_ROW0 4
#define KVC_ROW_CHUNKS 0   // chunks reserved so far
#define KVC_ROW_BASE 1     // first slot of the reserved chunk
#define KVC_ROW_FILLED 2   // slots filled (end of the reservation for LINEAR)
#define KVC_ROW_KVLEN 3    // active prefix attended by kvc_attend
__host__ __device__ inline int kvc_meta_row(int b) { return KVC_META_ROW0 + 4 * b; }
__host__ __device__ inline int kvc_meta_cu(int B) { return KVC_META_ROW0 + 4 * B; }

// A length layout shared by several handles: a caller-owned device block in the meta
// block's layout (error word, per-row kv_len, cu_seqlens) for `batch` rows.
struct kvc_lengths {
  int batch;
  int layout;     // KVC_LINEAR (kv_len) or KVC_PACKED (cu_seqlens)
  int cap;        // the largest length (LINEAR) or packed total it accepts
  int32_t* block;
};

struct kvc_cache {
  kvc_config cfg;
  int cap;            // slots per row (LINEAR capacity, CIRCULAR window) or packed total
  int eb;             // element bytes
  float scale;        // softmax scale
  void* k;
  void* v;
  int32_t* meta;
  const int32_t* lens;       // where attends and packed writes read kv_len / cu_seqlens:
                             // meta, or the block of a shared length layout (kvc_use_lengths)
  const kvc_lengths* bound;  // that shared layout, or null
  void* ws;
  int device;
  int num_sms;
  int dec_splits;     // split-KV decode: splits per (row, kv head); 0 = no decode kernel
  uint64_t debug_stall_ns;   // testing hook (kvc_debug_stall_waits); 0 in normal use
  bool tc_ok;         // the tensor-core chunk kernel serves this config
  CUtensorMap tm_k;   // K store, 128B-swizzled boxes of 64 dims x 128 slots (tensor-core kernel)
  CUtensorMap tm_v;   // V store, same boxes
  CUtensorMap tm_dk;  // K store, boxes of 64 dims x 64 slots (decode kernel)
  CUtensorMap tm_dv;  // V store, same boxes
};

// Row geometry of the store as seen by the attention kernels: row b's slot j lives
// at element ((b * row_stride_b) + (row0_b + j)) * Hkv * D + kvh * D.  For LINEAR
// and CIRCULAR row0_b = 0 and row_stride_b = cap; for PACKED row_stride_b = 0 and
// row0_b = cu_seqlens[b].
struct kvc_geom {
  int B, H, Hkv, D, cap, layout;
  const int32_t* lens;   // lengths block in the meta layout (the handle's meta or a shared layout)
};

// Valid slot range of row b, read on the device from the lengths block g.lens.
// Returns false (and sets the error word) when the row's length is out of range.
__device__ __forceinline__ bool kvc_row_range(const kvc_geom& g, int b, int* row0, int* len, int32_t* err_word) {
  const int32_t* meta = g.lens;
  if (g.layout == KVC_PACKED) {
    const int32_t* cu = meta + kvc_meta_cu(g.B);
    int lo = cu[b], hi = cu[b + 1];
    if (lo < 0 || hi <= lo || hi > g.cap) {
      atomicOr(err_word, KVC_DEV_BAD_CUSEQ);
      return false;
    }
    *row0 = lo;
    *len = hi - lo;
    return true;
  }
  int n = meta[kvc_meta_row(b) + KVC_ROW_KVLEN];
  if (n < 1 || n > g.cap) {
    atomicOr(err_word, KVC_DEV_BAD_KVLEN);
    return false;
  }
  *row0 = 0;
  *len = n;
  return true;
}

// Element offset of (row b, slot j, kv head kvh, dim 0).
__device__ __forceinline__ int64_t kvc_kv_offset(const kvc_geom& g, int b, int row0, int j, int kvh) {
  int64_t row = (g.layout == KVC_PACKED) ? (int64_t)(row0 + j) : (int64_t)b * g.cap + (row0 + j);
  return (row * g.Hkv + kvh) * (int64_t)g.D;
}

// ---- programmatic dependent launch ---------------------------------------------
// Kernels launched through kvc_launch_pdl may start (be scheduled, run their first
// instructions) while the previous kernel on the stream is still finishing; each of
// them calls kvc_pdl_wait() before it touches any global memory, which blocks until
// every prerequisite grid has completed and its writes are visible, so the stream
// order of the data is unchanged.  kvc_pdl_release() lets the next such kernel start.
__device__ __forceinline__ void kvc_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void kvc_pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t kvc_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Most splits the decode kernel takes per (row, kv head).
#define KVC_DECODE_MAX_SPLITS 1024

// ---- launchers (each returns a cudaError_t from the launch) ------------------
cudaError_t kvc_launch_advance(kvc_cache* c, int row, int n, cudaStream_t s);
cudaError_t kvc_launch_reset(kvc_cache* c, int row, cudaStream_t s);
cudaError_t kvc_launch_set_lengths(kvc_cache* c, const int32_t* kv_len, const int32_t* cu, cudaStream_t s);
cudaError_t kvc_launch_set_lengths_block(int32_t* block, int B, int cap, const int32_t* kv_len, const int32_t* cu,
                                         cudaStream_t s);
cudaError_t kvc_launch_write(kvc_cache* c, const void* k, const void* v, int n, const int32_t* slots,
                             cudaStream_t s);
cudaError_t kvc_launch_write_rope(kvc_cache* c, const void* k, const void* v, int n, const int32_t* slots,
                                  const float* rope, int rope_positions, cudaStream_t s);
cudaError_t kvc_launch_roll(kvc_cache* c, void* scratch, cudaStream_t s);
// One-launch append (reserve + write) of n tokens per row; only where kvc_append_fits.
bool kvc_append_fits(const kvc_cache* c, int n);
cudaError_t kvc_launch_append(kvc_cache* c, const void* k, const void* v, int n, cudaStream_t s);
cudaError_t kvc_launch_attn_simt(kvc_cache* c, const void* q, void* out, int n_q, bool causal, float* lse,
                                 cudaStream_t s);
cudaError_t kvc_launch_decode(kvc_cache* c, const void* q, void* out, float* lse, bool fixed_tiles, cudaStream_t s);
cudaError_t kvc_launch_decode_append(kvc_cache* c, const void* k_new, const void* v_new, const void* q, void* out,
                                     cudaStream_t s);
cudaError_t kvc_prepare_decode(kvc_cache* c);
bool kvc_decode_supported(const kvc_config& cfg);
int kvc_internal_check_config(const kvc_config* cfg, int* cap);
int kvc_internal_decode_splits(const kvc_config& cfg, int cap);
size_t kvc_decode_workspace_bytes(const kvc_config& cfg, int splits);
cudaError_t kvc_launch_attn_tc(kvc_cache* c, const void* q, void* out, int n_q, bool causal, float* lse,
                               cudaStream_t s);
cudaError_t kvc_launch_merge(int dtype, int rows, int head_dim, const void* oa, const float* la, const void* ob,
                             const float* lb, void* out, float* lse, cudaStream_t s);
bool kvc_tc_supported(const kvc_config& cfg);
bool kvc_tc_make_kv_maps(kvc_cache* c);
// Box shapes of a 4-D TMA map over a 16-bit tensor [d3][d2][d1][D] (D = 64 or 128):
//   KVC_BOX_SW128: 64 x 1 x box_rows x 1 elements, 128-byte swizzle (MMA operand tiles)
//   KVC_BOX_SW64:  32 x 1 x box_rows x 1, 64-byte swizzle (output staging of 32 columns)
enum kvc_box { KVC_BOX_SW128 = 0, KVC_BOX_SW64 = 2 };
// False if the driver entry point is missing or the encoding is rejected.
bool kvc_make_tile_map(CUtensorMap* m, int dtype, const void* base, int D, uint64_t d1, uint64_t d2, uint64_t d3,
                       uint32_t box_rows, kvc_box box = KVC_BOX_SW128);
// Decode maps of a store (tm_dk, tm_dv) for the config in c.
bool kvc_make_decode_maps(kvc_cache* c);
