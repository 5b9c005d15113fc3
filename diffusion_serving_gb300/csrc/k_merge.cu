// Merge of two attentions over disjoint key sets through their log-sum-exps (the
// forward_with_lse output of the TensorRT-LLM PR "FA4 variable-length cross-attention"
// makes split attention composable):
//   L = log(e^La + e^Lb),  o = e^(La - L) oa + e^(Lb - L) ob.
// A row whose both halves saw no key (La = Lb = -inf) gets L = -inf and o = 0.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace {

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__half* p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T>
__global__ void k_merge(int rows, int D, const T* __restrict__ oa, const float* __restrict__ la,
                        const T* __restrict__ ob, const float* __restrict__ lb, T* __restrict__ out,
                        float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const float a = la[r], b = lb[r];
    const float mx = fmaxf(a, b);
    float wa = 0.f, wb = 0.f, L = -INFINITY;
    if (mx != -INFINITY) {
      const float ea = expf(a - mx), eb = expf(b - mx);   // one of them is 1
      const float tot = ea + eb;
      L = mx + logf(tot);
      wa = ea / tot;
      wb = eb / tot;
    }
    for (int d = lane; d < D; d += 32)
      st(out + (int64_t)r * D + d, wa * ld(oa + (int64_t)r * D + d) + wb * ld(ob + (int64_t)r * D + d));
    if (lse != nullptr && lane == 0) lse[r] = L;
  }
}

}  // namespace

cudaError_t kvc_launch_merge(int dtype, int rows, int head_dim, const void* oa, const float* la, const void* ob,
                             const float* lb, void* out, float* lse, cudaStream_t s) {
  const int threads = 256;
  int blocks = (rows + threads / 32 - 1) / (threads / 32);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  switch (dtype) {
    case KVC_F32:
      k_merge<float><<<blocks, threads, 0, s>>>(rows, head_dim, (const float*)oa, la, (const float*)ob, lb,
                                                (float*)out, lse);
      break;
    case KVC_F16:
      k_merge<__half><<<blocks, threads, 0, s>>>(rows, head_dim, (const __half*)oa, la, (const __half*)ob, lb,
                                                 (__half*)out, lse);
      break;
    default:
      k_merge<__nv_bfloat16><<<blocks, threads, 0, s>>>(rows, head_dim, (const __nv_bfloat16*)oa, la,
                                                        (const __nv_bfloat16*)ob, lb, (__nv_bfloat16*)out, lse);
  }
  return cudaGetLastError();
}
