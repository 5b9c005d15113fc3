// Merge of two attentions over disjoint key sets through their log-sum-exps (the
// forward_with_lse output of the TensorRT-LLM PR "FA4 variable-length cross-attention"
// makes split attention composable):
//   L = log(e^La + e^Lb),  o = e^(La - L) oa + e^(Lb - L) ob.
// A row whose both halves saw no key (La = Lb = -inf) gets L = -inf and o = 0.
//
// HBM-bound (two rows read, one written, per output row).  Rows whose byte size is a
// power-of-two multiple of 16 with all three buffers 16-byte aligned take the vector
// kernel: one thread per 16-byte chunk of a row, kMergeUnroll chunks per thread loaded
// before any is combined, so every thread keeps 2 x kMergeUnroll 16-byte loads in
// flight.  Other shapes take the scalar kernel (a warp per row).  Both form the weights
// with the same expressions, so a row gets the same result from either, and both are
// launched as programmatic dependents (the launch overlaps the previous kernel's tail).
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeUnroll = 2;

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__half* p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// weights of the two halves and the merged LSE of one row: with mx the larger input,
// e^(La - mx) and e^(Lb - mx) are 1 and e = e^(-|La - Lb|), so one exponential, one
// logarithm and one reciprocal serve the row
__device__ __forceinline__ void merge_weights(float a, float b, float& wa, float& wb, float& L) {
  const float mx = fmaxf(a, b);
  wa = 0.f;
  wb = 0.f;
  L = -INFINITY;
  if (mx != -INFINITY) {
    const float e = expf(fminf(a, b) - mx);
    const float tot = 1.f + e;
    const float inv = 1.f / tot;
    L = mx + logf(tot);
    wa = a >= b ? inv : e * inv;
    wb = a >= b ? e * inv : inv;
  }
}

__device__ __forceinline__ float combine(float wa, float x, float wb, float y) {
  return __fmaf_rn(wa, x, __fmul_rn(wb, y));
}

template <typename T>
__global__ void __launch_bounds__(kMergeThreads)
k_merge(int rows, int D, const T* oa, const float* __restrict__ la, const T* ob, const float* __restrict__ lb,
        T* out, float* __restrict__ lse) {
  kvc_pdl_wait();
  kvc_pdl_release();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    float wa, wb, L;
    merge_weights(la[r], lb[r], wa, wb, L);
    for (int d = lane; d < D; d += 32)
      st(out + (int64_t)r * D + d, combine(wa, ld(oa + (int64_t)r * D + d), wb, ld(ob + (int64_t)r * D + d)));
    if (lse != nullptr && lane == 0) lse[r] = L;
  }
}

// 16 bytes of T as floats and back
template <typename T>
struct Chunk;
template <>
struct Chunk<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <typename H2, float2 (*ToF)(H2), H2 (*FromF)(float, float)>
struct Chunk16 {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      H2 h;
      memcpy(&h, &w[i], 4);
      const float2 x = ToF(h);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
  __device__ static uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const H2 h = FromF(f[2 * i], f[2 * i + 1]);
      memcpy(&w[i], &h, 4);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
__device__ __forceinline__ float2 h2_to_f2(__half2 h) { return __half22float2(h); }
__device__ __forceinline__ __half2 f2_to_h2(float a, float b) { return __floats2half2_rn(a, b); }
__device__ __forceinline__ float2 b2_to_f2(__nv_bfloat162 h) { return __bfloat1622float2(h); }
__device__ __forceinline__ __nv_bfloat162 f2_to_b2(float a, float b) { return __floats2bfloat162_rn(a, b); }
template <>
struct Chunk<__half> : Chunk16<__half2, h2_to_f2, f2_to_h2> {};
template <>
struct Chunk<__nv_bfloat16> : Chunk16<__nv_bfloat162, b2_to_f2, f2_to_b2> {};

// Chunk i of the flattened [rows, D] buffers belongs to row i >> row_shift (2^row_shift
// chunks per row).  Grid-stride over groups of kMergeUnroll chunks spaced one grid apart,
// so each of a group's loads is coalesced across the warp.
template <typename T>
__global__ void __launch_bounds__(kMergeThreads, 4)
k_merge_vec(int64_t chunks, int row_shift, const uint4* oa, const float* __restrict__ la, const uint4* ob,
            const float* __restrict__ lb, uint4* out, float* __restrict__ lse) {
  kvc_pdl_wait();
  kvc_pdl_release();
  using C = Chunk<T>;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t row_mask = ((int64_t)1 << row_shift) - 1;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < chunks; i0 += stride * kMergeUnroll) {
    uint4 va[kMergeUnroll], vb[kMergeUnroll];
    float a[kMergeUnroll], b[kMergeUnroll];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < chunks) {
        va[u] = oa[i];
        vb[u] = ob[i];
        a[u] = la[i >> row_shift];
        b[u] = lb[i >> row_shift];
      }
    }
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= chunks) break;
      float wa, wb, L;
      merge_weights(a[u], b[u], wa, wb, L);
      float x[C::N], y[C::N];
      C::unpack(va[u], x);
      C::unpack(vb[u], y);
#pragma unroll
      for (int e = 0; e < C::N; ++e) x[e] = combine(wa, x[e], wb, y[e]);
      out[i] = C::pack(x);
      if (lse != nullptr && (i & row_mask) == 0) lse[i >> row_shift] = L;
    }
  }
}

template <typename T>
cudaError_t launch_merge(int rows, int D, const void* oa, const float* la, const void* ob, const float* lb,
                         void* out, float* lse, cudaStream_t s) {
  const int64_t row_bytes = (int64_t)D * sizeof(T);
  const int64_t cpr = row_bytes / 16;   // 16-byte chunks per row
  const bool vec = row_bytes % 16 == 0 && (cpr & (cpr - 1)) == 0 && ((uintptr_t)oa % 16) == 0 &&
                   ((uintptr_t)ob % 16) == 0 && ((uintptr_t)out % 16) == 0;
  if (vec) {
    const int64_t chunks = (int64_t)rows * cpr;
    int64_t blocks = (chunks + (int64_t)kMergeThreads * kMergeUnroll - 1) / ((int64_t)kMergeThreads * kMergeUnroll);
    if (blocks > 152 * 64) blocks = 152 * 64;
    if (blocks < 1) blocks = 1;
    int shift = 0;   // log2 of the chunks per row
    for (int64_t n = cpr; n > 1; n >>= 1) ++shift;
    return kvc_launch_pdl(k_merge_vec<T>, dim3((unsigned)blocks), dim3(kMergeThreads), 0, s, chunks, shift,
                          (const uint4*)oa, la, (const uint4*)ob, lb, (uint4*)out, lse);
  }
  int blocks = (rows + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return kvc_launch_pdl(k_merge<T>, dim3(blocks), dim3(kMergeThreads), 0, s, rows, D, (const T*)oa, la, (const T*)ob,
                        lb, (T*)out, lse);
}

}  // namespace

cudaError_t kvc_launch_merge(int dtype, int rows, int head_dim, const void* oa, const float* la, const void* ob,
                             const float* lb, void* out, float* lse, cudaStream_t s) {
  switch (dtype) {
    case KVC_F32:
      return launch_merge<float>(rows, head_dim, oa, la, ob, lb, out, lse, s);
    case KVC_F16:
      return launch_merge<__half>(rows, head_dim, oa, la, ob, lb, out, lse, s);
    default:
      return launch_merge<__nv_bfloat16>(rows, head_dim, oa, la, ob, lb, out, lse, s);
  }
}
