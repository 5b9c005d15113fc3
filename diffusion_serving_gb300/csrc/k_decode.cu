// Split-KV decode attention: one query token per row over its active prefix.
//
// The decode step of the fish-speech PR "perf(text2semantic): pass only active KV
// cache prefix to SDPA" ("Change": decode step i attends kv_len = T + i + 1 slots,
// K/V sliced before head expansion).  The q heads of one GQA group share one read
// of their kv head's K and V (the repeat_interleave expansion of "Problem" is never
// materialised).  The query is the newest token, so no mask applies.
//
// Grid (splits, Hkv, B).  Each block takes an equal share of the row's kv_len slots
// (the share is computed on the device from kv_len, so the grid depends only on the
// capacity and a captured graph replays at any length), computes its G score rows
// into shared memory, their max and exp2 sums, then P.V, and writes an unnormalised
// partial (O_s, m_s, l_s) to the workspace.  The last block of each (b, kv head) to
// finish (a ticket counter in the workspace, left at zero for the next call) merges
// the partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
//
// Lane mapping: 8 lanes per slot row, each lane holding D/8 consecutive dims
// (16-byte vector loads), 4 slots per warp instruction.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTpsMax = 2048;   // most slots one block handles
constexpr int kUnroll = 4;      // slot groups with loads in flight per lane

__device__ __forceinline__ void unpack8(const uint4& u, float* f, const __half*) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 x = __half22float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
__device__ __forceinline__ void unpack8(const uint4& u, float* f, const __nv_bfloat16*) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 x = __bfloat1622float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
__device__ __forceinline__ void store_out(__half* p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads)
k_decode(const T* __restrict__ q, T* __restrict__ out, const T* __restrict__ kst, const T* __restrict__ vst,
         int32_t* __restrict__ meta, float* __restrict__ ws, kvc_geom g, float scale_log2) {
  constexpr int EPL = D / 8;      // dims per lane
  constexpr int VPL = EPL / 8;    // 16-byte vectors per lane
  extern __shared__ float smem[];
  float* sc = smem;                               // [G][kTpsMax] scores, then probabilities
  float* red = smem + G * kTpsMax;                // [kWarps][G][D] partial outputs
  __shared__ float s_m[G], s_l[G];
  __shared__ int s_last;

  const int split = blockIdx.x, nsplit = gridDim.x;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 7;        // dim slice
  const int grp = lane >> 3;       // slot within the warp's 4

  int row0 = 0, len = 0;
  if (!kvc_row_range(meta, g, b, &row0, &len, meta + KVC_META_ERR)) return;

  int tps = (len + nsplit - 1) / nsplit;
  tps = (tps + 15) & ~15;
  const int t0 = split * tps;
  const int t1 = min(len, t0 + tps);
  const int nt = max(0, t1 - t0);

  // query slice for this lane's dims, G heads, pre-scaled into the exp2 domain
  float qv[G][EPL];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    const T* qp = q + ((int64_t)b * g.H + kvh * G + gg) * D + sub * EPL;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      uint4 u = *reinterpret_cast<const uint4*>(qp + 8 * v);
      unpack8(u, &qv[gg][8 * v], (const T*)nullptr);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) qv[gg][e] *= scale_log2;
  }

  const int64_t row_step = (int64_t)g.Hkv * D;   // elements between consecutive slots
  const T* kbase = kst + kvc_kv_offset(g, b, row0, t0, kvh) + sub * EPL;
  const T* vbase = vst + kvc_kv_offset(g, b, row0, t0, kvh) + sub * EPL;

  // ---- scores ---------------------------------------------------------------
  // loop bounds are uniform per warp (the shuffles below need every lane)
  for (int tw = warp * 4; tw < nt; tw += kWarps * 4 * kUnroll) {
    const int tb = tw + grp;
    uint4 kr[kUnroll][VPL];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = tb + u * kWarps * 4;
      if (t < nt) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) kr[u][v] = __ldg(reinterpret_cast<const uint4*>(kbase + t * row_step) + v);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = tb + u * kWarps * 4;
      float kf[EPL];
#pragma unroll
      for (int v = 0; v < VPL; ++v) unpack8(kr[u][v], &kf[8 * v], (const T*)nullptr);
      float s[G];
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) a = fmaf(qv[gg][e], kf[e], a);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        s[gg] = a;
      }
      if (t < nt) {
#pragma unroll
        for (int gg = 0; gg < G; ++gg)
          if (sub == gg % 8) sc[gg * kTpsMax + t] = s[gg];
      }
    }
  }
  __syncthreads();

  // ---- softmax statistics per head -----------------------------------------
  for (int gg = warp; gg < G; gg += kWarps) {
    float mx = -INFINITY;
    for (int t = lane; t < nt; t += 32) mx = fmaxf(mx, sc[gg * kTpsMax + t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int t = lane; t < nt; t += 32) {
      const float p = exp2f(sc[gg * kTpsMax + t] - mx);
      sc[gg * kTpsMax + t] = p;
      sum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      s_m[gg] = mx;
      s_l[gg] = sum;
    }
  }
  __syncthreads();

  // ---- P.V ------------------------------------------------------------------
  float acc[G][EPL];
#pragma unroll
  for (int gg = 0; gg < G; ++gg)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[gg][e] = 0.f;
  for (int tw = warp * 4; tw < nt; tw += kWarps * 4 * kUnroll) {
    const int tb = tw + grp;
    uint4 vr[kUnroll][VPL];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = tb + u * kWarps * 4;
      if (t < nt) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) vr[u][v] = __ldg(reinterpret_cast<const uint4*>(vbase + t * row_step) + v);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = tb + u * kWarps * 4;
      if (t < nt) {
        float vf[EPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) unpack8(vr[u][v], &vf[8 * v], (const T*)nullptr);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float p = sc[gg * kTpsMax + t];
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[gg][e] = fmaf(p, vf[e], acc[gg][e]);
        }
      }
    }
  }
  // reduce the warp's 4 slot groups, then the warps through shared memory
#pragma unroll
  for (int gg = 0; gg < G; ++gg)
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float a = acc[gg][e];
      a += __shfl_xor_sync(0xffffffffu, a, 8);
      a += __shfl_xor_sync(0xffffffffu, a, 16);
      acc[gg][e] = a;
    }
  if (grp == 0) {
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int e = 0; e < EPL; ++e) red[(warp * G + gg) * D + sub * EPL + e] = acc[gg][e];
  }
  __syncthreads();

  const int pairs = g.B * g.Hkv;
  const int pair = b * g.Hkv + kvh;
  float* ws_o = ws;                                              // [pairs][nsplit][G][D]
  float* ws_ml = ws + (int64_t)pairs * nsplit * G * D;           // [pairs][nsplit][G][2]
  int* tickets = reinterpret_cast<int*>(ws_ml + (int64_t)pairs * nsplit * G * 2);  // [pairs]
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += red[w * G * D + e];
    ws_o[((int64_t)pair * nsplit + split) * G * D + e] = a;
  }
  if (threadIdx.x < G) {
    ws_ml[(((int64_t)pair * nsplit + split) * G + threadIdx.x) * 2 + 0] = s_m[threadIdx.x];
    ws_ml[(((int64_t)pair * nsplit + split) * G + threadIdx.x) * 2 + 1] = s_l[threadIdx.x];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(tickets + pair, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- merge the splits (last block of this (b, kv head)) -------------------
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int gg = e / D, d = e - gg * D;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2));
    float L = 0.f, o = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2);
      const float ls = __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2 + 1);
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      L = fmaf(w, ls, L);
      o = fmaf(w, __ldcg(ws_o + ((int64_t)pair * nsplit + s) * G * D + e), o);
    }
    store_out(out + ((int64_t)b * g.H + kvh * G + gg) * D + d, o / L);
  }
  if (threadIdx.x == 0) tickets[pair] = 0;
}

template <typename T, int D, int G>
cudaError_t launch_dg(kvc_cache* c, const void* q, void* out, cudaStream_t s, bool prepare_only) {
  const kvc_config& cfg = c->cfg;
  kvc_geom g{cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim, c->cap, cfg.layout};
  const size_t smem = (size_t)G * kTpsMax * 4 + (size_t)kWarps * G * D * 4;
  auto fn = k_decode<T, D, G>;
  if (prepare_only) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(c->dec_splits, cfg.kv_heads, cfg.batch);
  fn<<<grid, kThreads, smem, s>>>((const T*)q, (T*)out, (const T*)c->k, (const T*)c->v, c->meta, (float*)c->ws, g,
                                  c->scale * 1.4426950408889634f);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_d(kvc_cache* c, const void* q, void* out, cudaStream_t s, bool prep) {
  switch (c->cfg.heads / c->cfg.kv_heads) {
    case 1: return launch_dg<T, D, 1>(c, q, out, s, prep);
    case 2: return launch_dg<T, D, 2>(c, q, out, s, prep);
    case 4: return launch_dg<T, D, 4>(c, q, out, s, prep);
    default: return launch_dg<T, D, 8>(c, q, out, s, prep);
  }
}

template <typename T>
cudaError_t launch_t(kvc_cache* c, const void* q, void* out, cudaStream_t s, bool prep) {
  return c->cfg.head_dim == 64 ? launch_d<T, 64>(c, q, out, s, prep) : launch_d<T, 128>(c, q, out, s, prep);
}

}  // namespace

bool kvc_decode_supported(const kvc_config& cfg) {
  const int G = cfg.heads / cfg.kv_heads;
  return (cfg.dtype == KVC_F16 || cfg.dtype == KVC_BF16) && (cfg.head_dim == 64 || cfg.head_dim == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

size_t kvc_decode_workspace_bytes(const kvc_config& cfg, int splits) {
  const size_t pairs = (size_t)cfg.batch * cfg.kv_heads;
  const size_t G = cfg.heads / cfg.kv_heads;
  return pairs * splits * G * (cfg.head_dim + 2) * 4 + pairs * 4;
}

cudaError_t kvc_launch_decode(kvc_cache* c, const void* q, void* out, cudaStream_t s) {
  return c->cfg.dtype == KVC_F16 ? launch_t<__half>(c, q, out, s, false) : launch_t<__nv_bfloat16>(c, q, out, s, false);
}

// Opt the config's decode kernel into its dynamic shared memory (done at create time,
// so no attribute call happens while a stream is being captured).
cudaError_t kvc_prepare_decode(kvc_cache* c) {
  return c->cfg.dtype == KVC_F16 ? launch_t<__half>(c, nullptr, nullptr, 0, true)
                                 : launch_t<__nv_bfloat16>(c, nullptr, nullptr, 0, true);
}
