// fp32-FMA attention over the cache (any dtype, D = 64 or 128, any layout).
//
// out[b,i,h,:] = sum_j softmax_j(scale * q . k_j) v_j over row b's valid slots in
// physical order (flashdreams issue "add an opt-in circular KV policy for streaming
// attention", "proposed boundary": unmasked attention is invariant to permuting K
// and V rows together), restricted to the active prefix (fish-speech PR "pass only
// active KV cache prefix to SDPA", "Change") or the packed range (TensorRT-LLM PR
// "FA4 variable-length cross-attention", Description).  Causal (LINEAR only): the
// query at absolute position kv_len - n_q + i sees slots <= that position.
//
// Online softmax in the exp2 domain; scores, probabilities and accumulators are
// fp32 and every product is a true fp32 FMA (no TF32, no tensor cores).  This kernel
// serves fp32 stores and head dims the tensor-core kernel does not take, and is a
// cross-check of the other kernels.
//
// Block = 4 warps, one (b, h) and 16 query rows (4 per warp).  K/V tiles of 32 slots
// are staged in shared memory as fp32 (K rows padded by one word so that lane j
// reading row j is conflict-free).  In the score phase lane j owns slot j of the
// tile; in the PV phase lane l owns output dims l, l+32, ...
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 4;
constexpr int kRowsPerBlock = kRowsPerWarp * kWarps;
constexpr int kTile = 32;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
k_attn_simt(const T* __restrict__ q, T* __restrict__ out, const T* __restrict__ kst, const T* __restrict__ vst,
            int32_t* __restrict__ meta, kvc_geom g, int n_q, int causal, float scale_log2,
            float* __restrict__ lse) {
  constexpr int DL = D / 32;  // output dims per lane
  __shared__ float sK[kTile][D + 1];
  __shared__ float sV[kTile][D];
  __shared__ float sQ[kRowsPerBlock][D];

  kvc_pdl_wait();      // launched as a programmatic dependent: nothing is read before this
  kvc_pdl_release();
  const int b = blockIdx.z, h = blockIdx.y;
  const int i0 = blockIdx.x * kRowsPerBlock;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = h / (g.H / g.Hkv);

  int row0 = 0, len = 0;
  if (!kvc_row_range(g, b, &row0, &len, meta + KVC_META_ERR)) return;  // uniform per block

  // stage this block's query rows (pre-scaled into the exp2 domain)
  for (int e = threadIdx.x; e < kRowsPerBlock * D; e += blockDim.x) {
    const int r = e / D, d = e - r * D;
    const int i = i0 + r;
    float x = 0.f;
    if (i < n_q) x = to_f(q[(((int64_t)b * n_q + i) * g.H + h) * D + d]) * scale_log2;
    sQ[r][d] = x;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int t = 0; t < DL; ++t) acc[r][t] = 0.f;
  }
  const int qpos_base = len - n_q;  // absolute position of query 0 (causal)
  int kv_end = len;
  if (causal) {
    const int last = qpos_base + min(i0 + kRowsPerBlock, n_q) - 1;
    kv_end = min(len, last + 1);
  }

  for (int j0 = 0; j0 < kv_end; j0 += kTile) {
    __syncthreads();
    for (int e = threadIdx.x; e < kTile * D; e += blockDim.x) {
      const int j = e / D, d = e - j * D;
      float kx = 0.f, vx = 0.f;
      if (j0 + j < len) {
        const int64_t off = kvc_kv_offset(g, b, row0, j0 + j, kvh) + d;
        kx = to_f(kst[off]);
        vx = to_f(vst[off]);
      }
      sK[j][d] = kx;
      sV[j][d] = vx;
    }
    __syncthreads();

    // scores: lane owns slot j0 + lane for the warp's rows
    float s[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) s[r] = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      const float kd = sK[lane][d];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) s[r] = fmaf(sQ[warp * kRowsPerWarp + r][d], kd, s[r]);
    }
    const int j = j0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int i = i0 + warp * kRowsPerWarp + r;
      bool valid = j < len;
      if (causal) valid = valid && j <= qpos_base + i;
      float sv = valid ? s[r] : -INFINITY;
      float tmax = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float mnew = fmaxf(m[r], tmax);
      const float msafe = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = exp2f(m[r] - msafe);
      const float p = exp2f(sv - msafe);
      float psum = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[r] = l[r] * alpha + psum;
      m[r] = mnew;
#pragma unroll
      for (int t = 0; t < DL; ++t) acc[r][t] *= alpha;
      // PV: lane owns dims lane + 32 t
      for (int jj = 0; jj < kTile; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int t = 0; t < DL; ++t) acc[r][t] = fmaf(pj, sV[jj][lane + 32 * t], acc[r][t]);
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = i0 + warp * kRowsPerWarp + r;
    if (i >= n_q) continue;
    const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
    if (lse != nullptr && lane == 0)   // natural log of sum_j exp(scale q.k_j): m, l are in the exp2 domain
      lse[((int64_t)b * n_q + i) * g.H + h] = l[r] > 0.f ? (m[r] + log2f(l[r])) * 0.6931471805599453f : -INFINITY;
    T* o = out + (((int64_t)b * n_q + i) * g.H + h) * D;
#pragma unroll
    for (int t = 0; t < DL; ++t) o[lane + 32 * t] = from_f<T>(acc[r][t] * inv);
  }
}

template <typename T>
cudaError_t launch_t(kvc_cache* c, const void* q, void* out, int n_q, bool causal, float* lse, cudaStream_t s) {
  const kvc_config& cfg = c->cfg;
  kvc_geom g{cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim, c->cap, cfg.layout, c->lens};
  dim3 grid((n_q + kRowsPerBlock - 1) / kRowsPerBlock, cfg.heads, cfg.batch);
  const float sl2 = c->scale * 1.4426950408889634f;
  if (cfg.head_dim == 64)
    return kvc_launch_pdl(k_attn_simt<T, 64>, grid, dim3(kWarps * 32), 0, s, (const T*)q, (T*)out, (const T*)c->k,
                          (const T*)c->v, c->meta, g, n_q, causal ? 1 : 0, sl2, lse);
  return kvc_launch_pdl(k_attn_simt<T, 128>, grid, dim3(kWarps * 32), 0, s, (const T*)q, (T*)out, (const T*)c->k,
                        (const T*)c->v, c->meta, g, n_q, causal ? 1 : 0, sl2, lse);
}

}  // namespace

cudaError_t kvc_launch_attn_simt(kvc_cache* c, const void* q, void* out, int n_q, bool causal, float* lse,
                                 cudaStream_t s) {
  switch (c->cfg.dtype) {
    case KVC_F32: return launch_t<float>(c, q, out, n_q, causal, lse, s);
    case KVC_F16: return launch_t<__half>(c, q, out, n_q, causal, lse, s);
    default: return launch_t<__nv_bfloat16>(c, q, out, n_q, causal, lse, s);
  }
}
