// Cache bookkeeping and slot writes.
//
//  * k_advance   slot reservation for the next chunk (flashdreams issue "add an opt-in
//                circular KV policy for streaming attention", "proposed boundary":
//                reservation is separate from writes and lives in device memory).
//  * k_reset     row lifecycle reset (same section).
//  * k_set_lengths  active prefix kv_len (fish-speech PR "pass only active KV cache
//                prefix to SDPA", "Change") and packed offsets cu_seqlens (TensorRT-LLM
//                PR "FA4 variable-length cross-attention", Description).
//  * k_write     index_copy-style row scatter (lingbot-world PR "refactor(kv):
//                index_copy_ for KV-cache writes", Summary): bytes copied unchanged in
//                16-byte vectors, slot taken from device memory so replays of a
//                captured graph write the slot the device holds.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace {

__global__ void k_advance(int32_t* __restrict__ meta, int B, int row, int n, int layout, int sink,
                          int window, int chunk, int cap) {
  kvc_pdl_wait();
  kvc_pdl_release();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (row >= 0 && b != row) continue;
    int32_t* r = meta + kvc_meta_row(b);
    const int k = r[KVC_ROW_CHUNKS];
    if (layout == KVC_CIRCULAR) {
      const int64_t first = (int64_t)k * chunk;
      int base;
      if (first < window) {
        base = (int)first;                               // still filling
      } else {
        const int roll = (window - sink) / chunk;        // rolling chunks
        const int64_t idx = ((int64_t)k - sink / chunk) % roll;
        base = sink + (int)idx * chunk;                  // oldest rolling chunk
      }
      const int64_t filled = first + chunk < window ? first + chunk : window;
      r[KVC_ROW_CHUNKS] = k + 1;
      r[KVC_ROW_BASE] = base;
      r[KVC_ROW_FILLED] = (int)filled;
      r[KVC_ROW_KVLEN] = (int)filled;
    } else {  // LINEAR
      const int filled = r[KVC_ROW_FILLED];
      if ((int64_t)filled + n > cap) {
        atomicOr(meta + KVC_META_ERR, KVC_DEV_OVERFLOW);
        continue;
      }
      r[KVC_ROW_CHUNKS] = k + 1;
      r[KVC_ROW_BASE] = filled;
      r[KVC_ROW_FILLED] = filled + n;
      r[KVC_ROW_KVLEN] = filled + n;
    }
  }
}

__global__ void k_reset(int32_t* __restrict__ meta, int B, int row) {
  kvc_pdl_wait();
  kvc_pdl_release();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    if (row >= 0 && b != row) continue;
    int32_t* r = meta + kvc_meta_row(b);
    r[KVC_ROW_CHUNKS] = 0;
    r[KVC_ROW_BASE] = 0;
    r[KVC_ROW_FILLED] = 0;
    r[KVC_ROW_KVLEN] = 0;
  }
}

__global__ void k_set_lengths(int32_t* __restrict__ meta, int B, int cap, const int32_t* __restrict__ kv_len,
                              const int32_t* __restrict__ cu) {
  __shared__ int ok;
  kvc_pdl_wait();
  kvc_pdl_release();
  if (kv_len != nullptr) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int n = kv_len[b];
      if (n < 1 || n > cap) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_KVLEN);
      else meta[kvc_meta_row(b) + KVC_ROW_KVLEN] = n;
    }
  }
  if (cu == nullptr) return;
  if (threadIdx.x == 0) {
    int good = cu[0] == 0;
    for (int b = 0; b < B && good; ++b) good = cu[b + 1] > cu[b];
    good = good && cu[B] <= cap;
    ok = good;
    if (!good) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_CUSEQ);
  }
  __syncthreads();
  if (!ok) return;
  for (int b = threadIdx.x; b <= B; b += blockDim.x) meta[kvc_meta_cu(B) + b] = cu[b];
  for (int b = threadIdx.x; b < B; b += blockDim.x) meta[kvc_meta_row(b) + KVC_ROW_KVLEN] = cu[b + 1] - cu[b];
}

// One warp per (tensor, row b, token i): the warp resolves the destination row once,
// then its lanes copy the row's 16-byte vectors, 4 loads in flight per lane before
// the stores.  Destination row of (b, i):
//   slots given:  b * cap + slots[i]
//   reserved:     b * cap + base_b + i      (LINEAR also requires base_b + i < filled_b)
//   packed:       cu[b] + i for i < len_b (later tokens are padding and are skipped)
constexpr int kWriteThreads = 256;
constexpr int kWriteUnroll = 4;

__global__ void __launch_bounds__(kWriteThreads)
k_write(const uint4* __restrict__ ksrc, const uint4* __restrict__ vsrc, uint4* __restrict__ kdst,
        uint4* __restrict__ vdst, int32_t* __restrict__ meta, const int32_t* __restrict__ slots, int B, int n,
        int row_vecs, int cap, int layout) {
  kvc_pdl_wait();
  kvc_pdl_release();
  const int lane = threadIdx.x & 31;
  const int rows_per_tensor = B * n;
  const int rows = 2 * rows_per_tensor;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int t = r >= rows_per_tensor;
    const int e = r - (t ? rows_per_tensor : 0);
    const int b = e / n;
    const int i = e - b * n;
    int64_t drow = -1;
    if (layout == KVC_PACKED) {
      const int32_t* cu = meta + kvc_meta_cu(B);
      const int lo = cu[b], hi = cu[b + 1];
      if (i < hi - lo && lo >= 0 && hi <= cap) drow = lo + i;
    } else if (slots != nullptr) {
      const int s = slots[i];
      if (s >= 0 && s < cap) drow = (int64_t)b * cap + s;
      else if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_SLOT);
    } else {
      const int32_t* m = meta + kvc_meta_row(b);
      const int chunks = m[KVC_ROW_CHUNKS];
      const int s = m[KVC_ROW_BASE] + i;
      const bool ok = chunks > 0 && s >= 0 && s < cap && (layout != KVC_LINEAR || s < m[KVC_ROW_FILLED]);
      if (ok) drow = (int64_t)b * cap + s;
      else if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, chunks > 0 ? KVC_DEV_BAD_SLOT : KVC_DEV_NO_CHUNK);
    }
    if (drow < 0) continue;
    const uint4* src = (t ? vsrc : ksrc) + (int64_t)e * row_vecs;
    uint4* dst = (t ? vdst : kdst) + drow * row_vecs;
    for (int v0 = lane; v0 < row_vecs; v0 += 32 * kWriteUnroll) {
      uint4 val[kWriteUnroll];
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < row_vecs) val[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < row_vecs) dst[v] = val[u];
      }
    }
  }
}

// Write with RoPE fused into the K half: K rows are rotated at their absolute position
// before they are stored, V rows are copied unchanged (flashdreams issue "add an opt-in
// circular KV policy for streaming attention", "proposed boundary": absolute positions
// determine RoPE before storage).  Pair j of a head, (x[2j], x[2j+1]), turns by the
// angle whose (cos, sin) the caller's table holds at [pos][j]:
//   (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos), fp32 FMAs for 16-bit stores (fp64 for
//   fp32 stores), rounded once to the store type.
// Absolute position of token i: CIRCULAR (chunks - 1) * chunk + i; LINEAR base + i, or
// slots[i] when slots are given; PACKED i.  Rows whose position is outside the table
// are skipped and set KVC_DEV_BAD_POS.
template <typename T> struct Pack;
template <> struct Pack<__nv_bfloat16> {
  static constexpr int kPairs = 4;   // pairs per 16-byte vector
  __device__ static void rot(uint4& u, const float2* cs) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(h[i]);
      const float2 c = cs[i];
      h[i] = __floats2bfloat162_rn(fmaf(x.x, c.x, -x.y * c.y), fmaf(x.x, c.y, x.y * c.x));
    }
  }
};
template <> struct Pack<__half> {
  static constexpr int kPairs = 4;
  __device__ static void rot(uint4& u, const float2* cs) {
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __half22float2(h[i]);
      const float2 c = cs[i];
      h[i] = __floats2half2_rn(fmaf(x.x, c.x, -x.y * c.y), fmaf(x.x, c.y, x.y * c.x));
    }
  }
};
// fp32 stores turn the pair in fp64 and round once, so that the stored value is the
// correctly rounded rotation (fp32 arithmetic would leave ~1 ulp of its own rounding).
template <> struct Pack<float> {
  static constexpr int kPairs = 2;
  __device__ static void rot(uint4& u, const float2* cs) {
    float* f = reinterpret_cast<float*>(&u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const double x0 = f[2 * i], x1 = f[2 * i + 1];
      const double c = cs[i].x, sn = cs[i].y;
      f[2 * i] = (float)fma(x0, c, -x1 * sn);
      f[2 * i + 1] = (float)fma(x0, sn, x1 * c);
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kWriteThreads)
k_write_rope(const uint4* __restrict__ ksrc, const uint4* __restrict__ vsrc, uint4* __restrict__ kdst,
             uint4* __restrict__ vdst, int32_t* __restrict__ meta, const int32_t* __restrict__ slots,
             const float2* __restrict__ rope, int rope_positions, int B, int n, int row_vecs, int cap, int layout,
             int chunk, int head_dim) {
  constexpr int P = Pack<T>::kPairs;
  const int lane = threadIdx.x & 31;
  const int rows_per_tensor = B * n;
  const int rows = 2 * rows_per_tensor;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int half_d = head_dim / 2;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int t = r >= rows_per_tensor;
    const int e = r - (t ? rows_per_tensor : 0);
    const int b = e / n;
    const int i = e - b * n;
    int64_t drow = -1;
    int pos = -1;
    if (layout == KVC_PACKED) {
      const int32_t* cu = meta + kvc_meta_cu(B);
      const int lo = cu[b], hi = cu[b + 1];
      if (i < hi - lo && lo >= 0 && hi <= cap) drow = lo + i;
      pos = i;
    } else if (slots != nullptr) {
      const int sl = slots[i];
      if (sl >= 0 && sl < cap) drow = (int64_t)b * cap + sl;
      else if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_SLOT);
      pos = sl;
    } else {
      const int32_t* m = meta + kvc_meta_row(b);
      const int chunks = m[KVC_ROW_CHUNKS];
      const int sl = m[KVC_ROW_BASE] + i;
      const bool ok = chunks > 0 && sl >= 0 && sl < cap && (layout != KVC_LINEAR || sl < m[KVC_ROW_FILLED]);
      if (ok) drow = (int64_t)b * cap + sl;
      else if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, chunks > 0 ? KVC_DEV_BAD_SLOT : KVC_DEV_NO_CHUNK);
      pos = layout == KVC_CIRCULAR ? (chunks - 1) * chunk + i : sl;
    }
    if (drow < 0) continue;
    if (pos < 0 || pos >= rope_positions) {        // neither K nor V of such a token is written
      if (lane == 0 && t == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_BAD_POS);
      continue;
    }
    const uint4* src = (t ? vsrc : ksrc) + (int64_t)e * row_vecs;
    uint4* dst = (t ? vdst : kdst) + drow * row_vecs;
    const float2* cs_row = rope + (int64_t)pos * half_d;
    for (int v = lane; v < row_vecs; v += 32) {
      uint4 val = __ldg(src + v);
      if (t == 0) {
        const int pair0 = (v * P) % half_d;        // first pair of this vector within its head
        float2 cs[P];
#pragma unroll
        for (int k = 0; k < P; ++k) cs[k] = __ldg(cs_row + pair0 + k);
        Pack<T>::rot(val, cs);
      }
      dst[v] = val;
    }
  }
}

// Comparator for measurement, not on the path: the copy a chronological sink + window
// store makes once per chunk step (flashdreams issue "add an opt-in circular KV policy
// for streaming attention", "current path": the retained keys and values are cloned and
// copied back one chunk to the left).  Rows [first, first + count) of every batch row
// move between `src` (row stride src_cap) and `dst` (row stride dst_cap), K and V in
// one launch; the roll is two such launches: store -> scratch, scratch -> store.
__global__ void __launch_bounds__(kWriteThreads)
k_copy_rows(const uint4* __restrict__ ks, const uint4* __restrict__ vs, uint4* __restrict__ kd,
            uint4* __restrict__ vd, int B, int count, int src_cap, int src_first, int dst_cap, int dst_first,
            int row_vecs) {
  const int lane = threadIdx.x & 31;
  const int rows_per_tensor = B * count;
  const int rows = 2 * rows_per_tensor;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int t = r >= rows_per_tensor;
    const int e = r - (t ? rows_per_tensor : 0);
    const int b = e / count, i = e - b * count;
    const uint4* src = (t ? vs : ks) + ((int64_t)b * src_cap + src_first + i) * row_vecs;
    uint4* dst = (t ? vd : kd) + ((int64_t)b * dst_cap + dst_first + i) * row_vecs;
    for (int v0 = lane; v0 < row_vecs; v0 += 32 * kWriteUnroll) {
      uint4 val[kWriteUnroll];
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u)
        if (v0 + 32 * u < row_vecs) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u)
        if (v0 + 32 * u < row_vecs) dst[v0 + 32 * u] = val[u];
    }
  }
}

}  // namespace

cudaError_t kvc_launch_advance(kvc_cache* c, int row, int n, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  return kvc_launch_pdl(k_advance, dim3(1), dim3(128), 0, s, c->meta, g.batch, row, n, g.layout, g.sink, g.window,
                        g.chunk, c->cap);
}

cudaError_t kvc_launch_reset(kvc_cache* c, int row, cudaStream_t s) {
  return kvc_launch_pdl(k_reset, dim3(1), dim3(128), 0, s, c->meta, c->cfg.batch, row);
}

cudaError_t kvc_launch_set_lengths(kvc_cache* c, const int32_t* kv_len, const int32_t* cu, cudaStream_t s) {
  return kvc_launch_pdl(k_set_lengths, dim3(1), dim3(128), 0, s, c->meta, c->cfg.batch, c->cap, kv_len, cu);
}

cudaError_t kvc_launch_write(kvc_cache* c, const void* k, const void* v, int n, const int32_t* slots,
                             cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  const int64_t rows = 2LL * g.batch * n;
  int64_t blocks = (rows + kWriteThreads / 32 - 1) / (kWriteThreads / 32);
  const int64_t max_blocks = (int64_t)c->num_sms * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  return kvc_launch_pdl(k_write, dim3((unsigned)blocks), dim3(kWriteThreads), 0, s, (const uint4*)k, (const uint4*)v,
                        (uint4*)c->k, (uint4*)c->v, c->meta, slots, g.batch, n, row_vecs, c->cap, g.layout);
}

cudaError_t kvc_launch_write_rope(kvc_cache* c, const void* k, const void* v, int n, const int32_t* slots,
                                  const float* rope, int rope_positions, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  const int64_t rows = 2LL * g.batch * n;
  int64_t blocks = (rows + kWriteThreads / 32 - 1) / (kWriteThreads / 32);
  const int64_t max_blocks = (int64_t)c->num_sms * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
#define KVC_WR(T)                                                                                               \
  k_write_rope<T><<<(unsigned)blocks, kWriteThreads, 0, s>>>(                                                   \
      (const uint4*)k, (const uint4*)v, (uint4*)c->k, (uint4*)c->v, c->meta, slots, (const float2*)rope,         \
      rope_positions, g.batch, n, row_vecs, c->cap, g.layout, g.chunk, g.head_dim)
  if (g.dtype == KVC_F32) KVC_WR(float);
  else if (g.dtype == KVC_F16) KVC_WR(__half);
  else KVC_WR(__nv_bfloat16);
#undef KVC_WR
  return cudaGetLastError();
}

cudaError_t kvc_launch_roll(kvc_cache* c, void* scratch, cudaStream_t s) {
  const kvc_config& g = c->cfg;
  const int row_vecs = g.kv_heads * g.head_dim * c->eb / 16;
  const int count = g.window - g.sink - g.chunk;         // retained rolling tokens
  if (count <= 0) return cudaSuccess;
  const int64_t rows = 2LL * g.batch * count;
  int64_t blocks = (rows + kWriteThreads / 32 - 1) / (kWriteThreads / 32);
  const int64_t max_blocks = (int64_t)c->num_sms * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  uint4* sk = static_cast<uint4*>(scratch);
  uint4* sv = sk + (int64_t)g.batch * count * row_vecs;
  // clone: store rows [sink + chunk, window) -> scratch
  k_copy_rows<<<(unsigned)blocks, kWriteThreads, 0, s>>>((const uint4*)c->k, (const uint4*)c->v, sk, sv, g.batch,
                                                         count, c->cap, g.sink + g.chunk, count, 0, row_vecs);
  // copy back one chunk to the left: scratch -> store rows [sink, window - chunk)
  k_copy_rows<<<(unsigned)blocks, kWriteThreads, 0, s>>>(sk, sv, (uint4*)c->k, (uint4*)c->v, g.batch, count, count,
                                                         0, c->cap, g.sink, row_vecs);
  return cudaGetLastError();
}
