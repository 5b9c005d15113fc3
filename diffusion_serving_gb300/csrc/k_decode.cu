// Split-KV decode attention: one query token per row over its active prefix.
//
// The decode step of the fish-speech PR "perf(text2semantic): pass only active KV
// cache prefix to SDPA" ("Change": decode step i attends kv_len = T + i + 1 slots,
// K/V sliced before head expansion).  The q heads of one GQA group share one read
// of their kv head's K and V (the repeat_interleave expansion of "Problem" is never
// materialised).  The query is the newest token, so no mask applies.
//
// Grid (splits, Hkv, B).  Each block takes an equal share (at least kMinShare slots)
// of the row's kv_len slots; the share is computed on the device from kv_len, so the
// grid depends only on the shape and a captured graph replays at any length.
// Inside a block every warp streams its slots once, K and V of several slots in
// flight per lane, keeping an online softmax (running max m, sum l, accumulator) per
// q head; the warps' states merge in shared memory into one unnormalised partial
// (O_s, m_s, l_s) written to the workspace.  The last block of each (b, kv head) to
// finish (a ticket counter in the workspace, left at zero for the next call) merges
// the partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
//
// Lane mapping: 8 lanes per slot row, each lane holding D/8 consecutive dims
// (16-byte vector loads), 4 slots per warp instruction.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMinShare = 64;    // fewest slots a block takes (short prefixes use few splits)

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

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
k_decode(const T* __restrict__ q, T* __restrict__ out, const T* __restrict__ kst, const T* __restrict__ vst,
         int32_t* __restrict__ meta, float* __restrict__ ws, kvc_geom g, float scale_log2) {
  constexpr int EPL = D / 8;                     // dims per lane
  constexpr int VPL = EPL / 8;                   // 16-byte vectors per lane
  constexpr int U = (G * EPL > 64) ? 1 : 4;      // slot groups in flight per lane (register budget)
  constexpr int kStep = kWarps * 4;              // slots between a warp's consecutive groups
  __shared__ float s_acc[kWarps][G][D];
  __shared__ float s_ml[kWarps][G][2];
  __shared__ float s_red[kWarps];
  __shared__ float s_merge_w[KVC_DECODE_MAX_SPLITS];
  __shared__ int s_last;

  const int split = blockIdx.x, nsplit = gridDim.x;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 7;        // dim slice
  const int grp = lane >> 3;       // slot within the warp's 4

  int row0 = 0, len = 0;
  if (!kvc_row_range(meta, g, b, &row0, &len, meta + KVC_META_ERR)) return;

  int share = (len + nsplit - 1) / nsplit;
  share = max(share, kMinShare);
  share = (share + 15) & ~15;
  const int t0 = split * share;
  const int nt = max(0, min(len, t0 + share) - t0);

  // query slice for this lane's dims, G heads, pre-scaled into the exp2 domain
  float qv[G][EPL];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    const T* qp = q + ((int64_t)b * g.H + kvh * G + gg) * D + sub * EPL;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      uint4 u = __ldg(reinterpret_cast<const uint4*>(qp + 8 * v));
      unpack8(u, &qv[gg][8 * v], (const T*)nullptr);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) qv[gg][e] *= scale_log2;
  }

  const int64_t row_step = (int64_t)g.Hkv * D;   // elements between consecutive slots
  const T* kbase = kst + kvc_kv_offset(g, b, row0, t0, kvh) + sub * EPL;
  const T* vbase = vst + kvc_kv_offset(g, b, row0, t0, kvh) + sub * EPL;

  float m[G], l[G], acc[G][EPL];
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    m[gg] = -INFINITY;
    l[gg] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[gg][e] = 0.f;
  }

  // loop bounds are uniform per warp (the shuffles below need every lane)
  for (int tw = warp * 4; tw < nt; tw += kStep * U) {
    uint4 kr[U][VPL], vr[U][VPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tw + grp + u * kStep;
      if (t < nt) {
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
          kr[u][v] = __ldcs(reinterpret_cast<const uint4*>(kbase + t * row_step) + v);
          vr[u][v] = __ldcs(reinterpret_cast<const uint4*>(vbase + t * row_step) + v);
        }
      } else {
#pragma unroll
        for (int v = 0; v < VPL; ++v) kr[u][v] = vr[u][v] = make_uint4(0, 0, 0, 0);
      }
    }
    float s[U][G];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[EPL];
#pragma unroll
      for (int v = 0; v < VPL; ++v) unpack8(kr[u][v], &kf[8 * v], (const T*)nullptr);
      const bool valid = tw + grp + u * kStep < nt;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) a = fmaf(qv[gg][e], kf[e], a);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        s[u][gg] = valid ? a : -INFINITY;
      }
    }
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      float mx = s[0][gg];
#pragma unroll
      for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[u][gg]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      // finite: slot tw (group 0, u = 0) is valid on every pass of this loop
      const float mnew = fmaxf(m[gg], mx);
      const float alpha = ex2(m[gg] - mnew);
      m[gg] = mnew;
      l[gg] *= alpha;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[gg][e] *= alpha;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = ex2(s[u][gg] - mnew);
        l[gg] += p;
        float vf[EPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) unpack8(vr[u][v], &vf[8 * v], (const T*)nullptr);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[gg][e] = fmaf(p, vf[e], acc[gg][e]);
      }
    }
  }
  // Sum the warp's 4 slot groups (they share m).  Every lane of a group added the
  // same p values to l, so after the sum any lane holds the warp's total.
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    l[gg] += __shfl_xor_sync(0xffffffffu, l[gg], 8);
    l[gg] += __shfl_xor_sync(0xffffffffu, l[gg], 16);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float a = acc[gg][e];
      a += __shfl_xor_sync(0xffffffffu, a, 8);
      a += __shfl_xor_sync(0xffffffffu, a, 16);
      acc[gg][e] = a;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) s_acc[warp][gg][sub * EPL + e] = acc[gg][e];
      if (sub == 0) {
        s_ml[warp][gg][0] = m[gg];
        s_ml[warp][gg][1] = l[gg];
      }
    }
  }
  __syncthreads();

  // ---- this block's partial: merge the warps ---------------------------------
  const int pairs = g.B * g.Hkv;
  const int pair = b * g.Hkv + kvh;
  float* ws_o = ws;                                              // [pairs][nsplit][G][D]
  float* ws_ml = ws + (int64_t)pairs * nsplit * G * D;           // [pairs][nsplit][G][2]
  int* tickets = reinterpret_cast<int*>(ws_ml + (int64_t)pairs * nsplit * G * 2);  // [pairs]
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int gg = e / D, d = e - gg * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][gg][0]);
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = s_ml[w][gg][0];
      if (mw != -INFINITY) a = fmaf(ex2(mw - M), s_acc[w][gg][d], a);
    }
    ws_o[((int64_t)pair * nsplit + split) * G * D + e] = a;
  }
  if (threadIdx.x < G) {
    const int gg = threadIdx.x;
    float M = -INFINITY, L = 0.f;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][gg][0]);
    for (int w = 0; w < kWarps; ++w) {
      const float mw = s_ml[w][gg][0];
      if (mw != -INFINITY) L = fmaf(ex2(mw - M), s_ml[w][gg][1], L);
    }
    ws_ml[(((int64_t)pair * nsplit + split) * G + gg) * 2 + 0] = M;
    ws_ml[(((int64_t)pair * nsplit + split) * G + gg) * 2 + 1] = L;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(tickets + pair, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- merge the splits (last block of this (b, kv head)) -------------------
  const int used = min(nsplit, (len + share - 1) / share);       // later splits are empty
  for (int gg = 0; gg < G; ++gg) {
    float M = -INFINITY;
    for (int s = threadIdx.x; s < used; s += blockDim.x)
      M = fmaxf(M, __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) s_red[warp] = M;
    __syncthreads();
    M = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_red[w]);
    __syncthreads();
    float L = 0.f;
    for (int s = threadIdx.x; s < used; s += blockDim.x) {
      const float ms = __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2);
      const float ls = __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2 + 1);
      const float wgt = ms == -INFINITY ? 0.f : ex2(ms - M);
      s_merge_w[s] = wgt;
      L = fmaf(wgt, ls, L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) s_red[warp] = L;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += s_red[w];
    const float inv = 1.f / tot;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      float o0 = 0.f, o1 = 0.f;
      int s = 0;
      for (; s + 1 < used; s += 2) {
        o0 = fmaf(s_merge_w[s], __ldcg(ws_o + (((int64_t)pair * nsplit + s) * G + gg) * D + d), o0);
        o1 = fmaf(s_merge_w[s + 1], __ldcg(ws_o + (((int64_t)pair * nsplit + s + 1) * G + gg) * D + d), o1);
      }
      if (s < used) o0 = fmaf(s_merge_w[s], __ldcg(ws_o + (((int64_t)pair * nsplit + s) * G + gg) * D + d), o0);
      store_out(out + ((int64_t)b * g.H + kvh * G + gg) * D + d, (o0 + o1) * inv);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) tickets[pair] = 0;
}

template <typename T, int D, int G>
cudaError_t launch_dg(kvc_cache* c, const void* q, void* out, cudaStream_t s) {
  const kvc_config& cfg = c->cfg;
  kvc_geom g{cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim, c->cap, cfg.layout};
  dim3 grid(c->dec_splits, cfg.kv_heads, cfg.batch);
  k_decode<T, D, G><<<grid, kThreads, 0, s>>>((const T*)q, (T*)out, (const T*)c->k, (const T*)c->v, c->meta,
                                              (float*)c->ws, g, c->scale * 1.4426950408889634f);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_d(kvc_cache* c, const void* q, void* out, cudaStream_t s) {
  switch (c->cfg.heads / c->cfg.kv_heads) {
    case 1: return launch_dg<T, D, 1>(c, q, out, s);
    case 2: return launch_dg<T, D, 2>(c, q, out, s);
    case 4: return launch_dg<T, D, 4>(c, q, out, s);
    default: return launch_dg<T, D, 8>(c, q, out, s);
  }
}

template <typename T>
cudaError_t launch_t(kvc_cache* c, const void* q, void* out, cudaStream_t s) {
  return c->cfg.head_dim == 64 ? launch_d<T, 64>(c, q, out, s) : launch_d<T, 128>(c, q, out, s);
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
  return c->cfg.dtype == KVC_F16 ? launch_t<__half>(c, q, out, s) : launch_t<__nv_bfloat16>(c, q, out, s);
}

// ---------------------------------------------------------------------------
// Allocation-free decode entry point.
//
// Some callers cannot allocate device memory at all: code running inside another
// framework's memory pool, plugins whose host process owns every cudaMalloc, or
// steps that must not allocate once a graph has been captured.  They still own the
// K/V stores, the meta block, the query and the output, but have nowhere to put the
// decode kernel's scratch (per-split partial outputs and the per-(row, kv head)
// tickets).  kvc_attend_decode_noalloc gives them the same decode kernel with that
// scratch in a fixed array compiled into this library: kDecodeScratchBytes (4 MiB)
// of device memory that every GPU which loads the library holds until the process
// exits.  All calls share it, so calls that overlap on the GPU (different streams,
// or different host threads without ordering) race on it; calls on one stream are
// ordered and safe.  It keeps the last call's contents; the tickets, which must
// start at zero, are cleared by every call.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kDecodeScratchBytes = 4u << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

// Device address of g_decode_scratch, looked up once per device with that device
// current.  In host code the array's name is only a stand-in for the symbol, never
// a pointer a kernel may be given.
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int kvc_attend_decode_noalloc(const kvc_config* cfg, const void* k_store, const void* v_store,
                                         int32_t* meta, const void* q, void* out, void* stream) {
  int cap = 0;
  const int rc = kvc_internal_check_config(cfg, &cap);
  if (rc != KVC_OK) return rc;
  if (!kvc_decode_supported(*cfg)) return KVC_ERR_UNSUPPORTED;
  const uintptr_t mis = (uintptr_t)k_store | (uintptr_t)v_store | (uintptr_t)meta | (uintptr_t)q | (uintptr_t)out;
  if (!k_store || !v_store || !meta || !q || !out || (mis & 15u)) return KVC_ERR_ARG;
  const int splits = kvc_internal_decode_splits(*cfg, cap);
  const size_t need = kvc_decode_workspace_bytes(*cfg, splits);
  if (need > kDecodeScratchBytes) return KVC_ERR_RANGE;   // too many (row, kv head) pairs for the array
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return KVC_ERR_CUDA;

  // the same kernel as kvc_attend's decode path, on a handle that lives on this stack
  kvc_cache c{};
  c.cfg = *cfg;
  c.cap = cap;
  c.eb = 2;
  c.scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0f / sqrtf((float)cfg->head_dim);
  c.k = const_cast<void*>(k_store);
  c.v = const_cast<void*>(v_store);
  c.meta = meta;
  c.ws = scratch;
  c.dec_splits = splits;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the tickets sit after the partials; an earlier call with another shape may have
  // left partial data there
  const size_t pairs = (size_t)cfg->batch * cfg->kv_heads;
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - pairs * 4), 0, pairs * 4, s) != cudaSuccess)
    return KVC_ERR_CUDA;
  return kvc_launch_decode(&c, q, out, s) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}
