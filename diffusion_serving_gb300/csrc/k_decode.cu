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
// A producer warp streams the share through a ring of shared-memory stages with TMA
// tile loads (112 whole rows of one kv head per box): one instruction moves 28 KB of K
// or V, so the whole stream needs a few hundred copy requests per SM.  Seven consumer
// warps take 16 slots of every 112-slot tile each, as 4 independent row groups whose
// loads and dot products overlap and keep an online softmax (running
// max m, sum l, accumulator) per q head; their states merge in shared memory into one
// unnormalised partial (O_s, m_s, l_s) written to the workspace.  The last block of
// each (b, kv head) to finish (a ticket counter in the workspace, left at zero for the
// next call) merges the partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
//
// Lane mapping: 8 lanes per slot row, 4 rows per warp instruction; lane sub holds dims
// {64 v + 8 sub + i : v < D/64, i < 8}, i.e. 16-byte chunk `sub` of each 64-dim half, so
// the 8 lanes of a row read 128 contiguous bytes per load (one wavefront per row).
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

namespace {

// 8 warps per block: registers are split over the SM's 4 sub-partitions, so a block of
// 8 warps may give each thread up to 255 registers (9 warps would cap it at 168).
constexpr int kWarps = 7;                   // consumer warps
constexpr int kGroups = 4;                  // row groups of 4 per consumer warp per tile
constexpr int kRowsPerWarp = kGroups * 4;   // 16 rows of every tile per consumer warp
constexpr int kThreads = (kWarps + 1) * 32; // + one producer warp
constexpr int kMinShare = 64;               // fewest slots a block takes (short prefixes use few splits)
constexpr int kTile = kWarps * kRowsPerWarp;  // 112 slots per stage (one TMA box of rows: 14 swizzle atoms)
constexpr int kStages = 3;                  // 3 x 56 KB in flight per SM (bandwidth x latency)
constexpr uint64_t kTimeoutNs = 500000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait (0.5 s of %globaltimer); false when it ran out or the block is aborting.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (honour_abort && *abort) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

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

template <int D>
__host__ __device__ constexpr uint32_t box_bytes() { return kTile * D * 2u; }         // kTile whole rows
template <int D>
__host__ __device__ constexpr uint32_t stage_bytes() { return 2u * box_bytes<D>(); }  // K and V
template <int D>
__host__ __device__ constexpr size_t dyn_smem_bytes() { return (size_t)kStages * stage_bytes<D>() + 1024; }

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
k_decode(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const T* __restrict__ q,
         T* __restrict__ out, int32_t* __restrict__ meta, float* __restrict__ ws, kvc_geom g, float scale_log2,
         float* __restrict__ lse) {
  constexpr int VPL = D / 64;        // 16-byte vectors (= 64-dim boxes) per lane per row
  constexpr int EPL = VPL * 8;       // dims per lane
  constexpr uint32_t BOX = box_bytes<D>();
  constexpr uint32_t SB = stage_bytes<D>();
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ float s_acc[kWarps][G][D];
  __shared__ float s_ml[kWarps][G][2];
  __shared__ float s_inv[G];
  __shared__ int s_last, s_abort;

  const int split = blockIdx.x, nsplit = gridDim.x;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane & 7;          // dim slice
  const int grp = lane >> 3;         // row within the group of 4

  kvc_pdl_wait();
  kvc_pdl_release();
  int row0 = 0, len = 0;
  if (!kvc_row_range(meta, g, b, &row0, &len, meta + KVC_META_ERR)) return;

  int share = (len + nsplit - 1) / nsplit;
  share = max(share, kMinShare);
  share = (share + 15) & ~15;
  const int t0 = split * share;
  const int nt = max(0, min(len, t0 + share) - t0);
  const int n_tiles = (nt + kTile - 1) / kTile;

  if (threadIdx.x < kStages) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], kWarps);
  }
  if (threadIdx.x == 0) s_abort = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  volatile int* abort = &s_abort;

  if (warp == kWarps) {
    // ---------------- producer: TMA tiles of K and V into the stage ring ----------------
    if (lane == 0) {
      const int kv_batch = g.layout == KVC_PACKED ? 0 : b;
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % kStages;
        if (t >= kStages && !mbar_wait(&empty[st], ((t / kStages) - 1) & 1, abort)) break;
        mbar_expect_tx(&full[st], SB);
        uint8_t* dst = dsm + st * SB;
        const int row = row0 + t0 + t * kTile;
        tma_load_4d(&tm_k, &full[st], dst, 0, kvh, row, kv_batch);
        tma_load_4d(&tm_v, &full[st], dst + BOX, 0, kvh, row, kv_batch);
        issued = t + 1;
      }
      if (*abort) {   // let every load issued here land before the block releases its shared memory
        for (int t = max(0, issued - kStages); t < issued; ++t)
          mbar_wait(&full[t % kStages], (t / kStages) & 1, abort, false);
      }
    }
  }

  // query slice for this lane's dims, G heads, pre-scaled into the exp2 domain
  float qv[G][EPL];
  float m[G], l[G], acc[G][EPL];
  if (warp < kWarps) {
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const T* qp = q + ((int64_t)b * g.H + kvh * G + gg) * D;
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        uint4 u = __ldg(reinterpret_cast<const uint4*>(qp + 64 * v + 8 * sub));
        unpack8(u, &qv[gg][8 * v], (const T*)nullptr);
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) qv[gg][e] *= scale_log2;
      m[gg] = -INFINITY;
      l[gg] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[gg][e] = 0.f;
    }

    for (int t = 0; t < n_tiles; ++t) {
      const int st = t % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (t / kStages) & 1, abort))) break;
      const uint8_t* kst = dsm + st * SB;
      const uint8_t* vst = kst + BOX;
      const int first = t * kTile + warp * kRowsPerWarp;   // this warp's rows of the tile
      if (first < nt) {
        // scores of the warp's kGroups row groups (independent: they overlap in flight)
        float sc[kGroups][G];
#pragma unroll
        for (int u = 0; u < kGroups; ++u) {
          const int r = warp * kRowsPerWarp + u * 4 + grp;          // row within the tile
          const uint32_t off = r * (D * 2) + sub * 16;                // 16-byte chunk `sub` of each 64-dim half
          float kf[EPL];
#pragma unroll
          for (int v = 0; v < VPL; ++v)
            unpack8(*reinterpret_cast<const uint4*>(kst + off + v * 128), &kf[8 * v], (const T*)nullptr);
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EPL; e += 2)
              a2 = __ffma2_rn(make_float2(qv[gg][e], qv[gg][e + 1]), make_float2(kf[e], kf[e + 1]), a2);
            sc[u][gg] = a2.x + a2.y;
          }
        }
#pragma unroll
        for (int u = 0; u < kGroups; ++u)
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            float a = sc[u][gg];
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            sc[u][gg] = first + u * 4 + grp < nt ? a : -INFINITY;
          }
        // online softmax update per head, then P.V with V re-read from shared memory
        float p[kGroups][G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          float mx = sc[0][gg];
#pragma unroll
          for (int u = 1; u < kGroups; ++u) mx = fmaxf(mx, sc[u][gg]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          if (mx > m[gg]) {                                // warp-uniform: the running max grows
            const float alpha = ex2(m[gg] - mx);           // 0 on the first tile (m = -inf)
            m[gg] = mx;
            l[gg] *= alpha;
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
              const float2 y = __fmul2_rn(make_float2(acc[gg][e], acc[gg][e + 1]), make_float2(alpha, alpha));
              acc[gg][e] = y.x;
              acc[gg][e + 1] = y.y;
            }
          }
#pragma unroll
          for (int u = 0; u < kGroups; ++u) {
            p[u][gg] = ex2(sc[u][gg] - m[gg]);
            l[gg] += p[u][gg];
          }
        }
        const bool partial = first + kRowsPerWarp > nt;     // stale rows past nt: their V is zeroed
#pragma unroll
        for (int u = 0; u < kGroups; ++u) {
          const int r = warp * kRowsPerWarp + u * 4 + grp;
          const uint32_t off = r * (D * 2) + sub * 16;
          float vf[EPL];
#pragma unroll
          for (int v = 0; v < VPL; ++v)
            unpack8(*reinterpret_cast<const uint4*>(vst + off + v * 128), &vf[8 * v], (const T*)nullptr);
          if (partial && first + u * 4 + grp >= nt) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) vf[e] = 0.f;
          }
#pragma unroll
          for (int gg = 0; gg < G; ++gg)
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
              const float2 y = __ffma2_rn(make_float2(p[u][gg], p[u][gg]), make_float2(vf[e], vf[e + 1]),
                                          make_float2(acc[gg][e], acc[gg][e + 1]));
              acc[gg][e] = y.x;
              acc[gg][e + 1] = y.y;
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);           // this warp is done with the stage
    }
    // Sum the warp's 4 row groups (they share m).  Every lane of a group added the same
    // p values to l, so after the sum any lane holds the warp's total.
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
        for (int e = 0; e < EPL; ++e) s_acc[warp][gg][(e >> 3) * 64 + sub * 8 + (e & 7)] = acc[gg][e];
        if (sub == 0) {
          s_ml[warp][gg][0] = m[gg];
          s_ml[warp][gg][1] = l[gg];
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) atomicOr(meta + KVC_META_ERR, KVC_DEV_TIMEOUT);

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
  // (m_s, l_s) of every used split and head into shared memory (the stage ring is free
  // now), weights 2^(m_s - M) per head, then O over the splits.
  const int used = min(nsplit, (len + share - 1) / share);       // later splits are empty
  float* sw = reinterpret_cast<float*>(dsm);                     // [G][used] weights
  float* sl = sw + G * used;                                     // [G][used] sums
  for (int e = threadIdx.x; e < G * used; e += blockDim.x) {
    const int gg = e / used, s = e - gg * used;
    sw[e] = __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2);
    sl[e] = __ldcg(ws_ml + (((int64_t)pair * nsplit + s) * G + gg) * 2 + 1);
  }
  __syncthreads();
  for (int gg = warp; gg < G; gg += kWarps + 1) {
    float M = -INFINITY;
    for (int s = lane; s < used; s += 32) M = fmaxf(M, sw[gg * used + s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int s = lane; s < used; s += 32) {
      const float ms = sw[gg * used + s];
      const float wgt = ms == -INFINITY ? 0.f : ex2(ms - M);
      sw[gg * used + s] = wgt;
      L = fmaf(wgt, sl[gg * used + s], L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      s_inv[gg] = 1.f / L;
      if (lse != nullptr) lse[(int64_t)b * g.H + kvh * G + gg] = (M + log2f(L)) * 0.6931471805599453f;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int gg = e / D, d = e - gg * D;
    const float* wrow = sw + gg * used;
    const float* src = ws_o + (int64_t)pair * nsplit * G * D + (int64_t)gg * D + d;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    int s = 0;
    for (; s + 3 < used; s += 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = fmaf(wrow[s + k], __ldcg(src + (int64_t)(s + k) * G * D), o[k]);
    }
    for (; s < used; ++s) o[0] = fmaf(wrow[s], __ldcg(src + (int64_t)s * G * D), o[0]);
    store_out(out + ((int64_t)b * g.H + kvh * G + gg) * D + d, ((o[0] + o[1]) + (o[2] + o[3])) * s_inv[gg]);
  }
  if (threadIdx.x == 0) tickets[pair] = 0;
}

template <typename T, int D, int G>
cudaError_t launch_dg(kvc_cache* c, const void* q, void* out, float* lse, cudaStream_t s, bool prepare) {
  constexpr size_t smem = dyn_smem_bytes<D>();
  if (prepare) return cudaFuncSetAttribute(k_decode<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const kvc_config& cfg = c->cfg;
  kvc_geom g{cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim, c->cap, cfg.layout};
  dim3 grid(c->dec_splits, cfg.kv_heads, cfg.batch);
  return kvc_launch_pdl(k_decode<T, D, G>, grid, dim3(kThreads), smem, s, c->tm_dk, c->tm_dv, (const T*)q, (T*)out,
                        c->meta, (float*)c->ws, g, c->scale * 1.4426950408889634f, lse);
}

template <typename T, int D>
cudaError_t launch_d(kvc_cache* c, const void* q, void* out, float* lse, cudaStream_t s, bool prepare) {
  switch (c->cfg.heads / c->cfg.kv_heads) {
    case 1: return launch_dg<T, D, 1>(c, q, out, lse, s, prepare);
    case 2: return launch_dg<T, D, 2>(c, q, out, lse, s, prepare);
    case 4: return launch_dg<T, D, 4>(c, q, out, lse, s, prepare);
    default: return launch_dg<T, D, 8>(c, q, out, lse, s, prepare);
  }
}

template <typename T>
cudaError_t launch_t(kvc_cache* c, const void* q, void* out, float* lse, cudaStream_t s, bool prepare) {
  return c->cfg.head_dim == 64 ? launch_d<T, 64>(c, q, out, lse, s, prepare)
                               : launch_d<T, 128>(c, q, out, lse, s, prepare);
}

// The decode kernels opt into their dynamic shared memory once per process and
// device, before their first launch.
std::mutex g_prep_mu;
bool g_prepared[64][2][2][4];

cudaError_t prepare_once(kvc_cache* c) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int ti = c->cfg.dtype == KVC_F16 ? 0 : 1, di = c->cfg.head_dim == 64 ? 0 : 1;
  const int G = c->cfg.heads / c->cfg.kv_heads;
  const int gi = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lock(g_prep_mu);
  if (g_prepared[dev][ti][di][gi]) return cudaSuccess;
  e = ti == 0 ? launch_t<__half>(c, nullptr, nullptr, nullptr, 0, true)
              : launch_t<__nv_bfloat16>(c, nullptr, nullptr, nullptr, 0, true);
  if (e == cudaSuccess) g_prepared[dev][ti][di][gi] = true;
  return e;
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

cudaError_t kvc_prepare_decode(kvc_cache* c) { return prepare_once(c); }

bool kvc_make_decode_maps(kvc_cache* c) {
  const kvc_config& g = c->cfg;
  const uint64_t batches = g.layout == KVC_PACKED ? 1 : (uint64_t)g.batch;
  const uint64_t cap = (uint64_t)c->cap;
  return kvc_make_tile_map(&c->tm_dk, g.dtype, c->k, g.head_dim, g.kv_heads, cap, batches, kTile, KVC_BOX_ROWS) &&
         kvc_make_tile_map(&c->tm_dv, g.dtype, c->v, g.head_dim, g.kv_heads, cap, batches, kTile, KVC_BOX_ROWS);
}

cudaError_t kvc_launch_decode(kvc_cache* c, const void* q, void* out, float* lse, cudaStream_t s) {
  const cudaError_t e = prepare_once(c);
  if (e != cudaSuccess) return e;
  return c->cfg.dtype == KVC_F16 ? launch_t<__half>(c, q, out, lse, s, false)
                                 : launch_t<__nv_bfloat16>(c, q, out, lse, s, false);
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
  if (!kvc_make_decode_maps(&c)) return KVC_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the tickets sit after the partials; an earlier call with another shape may have
  // left partial data there
  const size_t pairs = (size_t)cfg->batch * cfg->kv_heads;
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - pairs * 4), 0, pairs * 4, s) != cudaSuccess)
    return KVC_ERR_CUDA;
  return kvc_launch_decode(&c, q, out, nullptr, s) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}
