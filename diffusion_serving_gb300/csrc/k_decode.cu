// Split-KV decode attention: one query token per row over its active prefix.
//
// The decode step of the fish-speech PR "perf(text2semantic): pass only active KV
// cache prefix to SDPA" ("Change": decode step i attends kv_len = T + i + 1 slots,
// K/V sliced before head expansion).  The q heads of one GQA group share one read
// of their kv head's K and V (the repeat_interleave expansion of "Problem" is never
// materialised).  The query is the newest token, so no mask applies.
//
// Grid (splits, Hkv, B); the grid depends only on the shape, so a captured graph
// replays at any length.  A block takes its (row, kv head) pair and its split from its
// linear launch index, pairs interleaved.  A row's kv_len slots form tiles of kTile
// slots.  A row of at most kSoloTiles tiles (kSoloTilesAppend in the append
// instantiation) is streamed by one block, which writes the output directly.
// Otherwise each block streams some of its (row, kv head)'s tiles: kStages fixed ones
// first, then tiles claimed one at a time from a counter, so faster blocks take more.  A producer warp
// moves each tile into a ring of shared-memory stages with TMA (128-byte-swizzled
// boxes of 64 dims x kTile slots, K and V).  Seven consumer warps take 16 slots of
// every tile each: S = Q K^T and O += P V run as warp-level m16n8k16 MMAs (the G q
// heads of the group in M, padded to 16; slots or dims in N), with an online softmax
// (running max m, sum l) per head row in between.  The warps' states merge in shared
// memory into one unnormalised partial (O_s, m_s, l_s) per block, written to the
// workspace; the last block of each (row, kv head) to finish (a ticket counter, left
// at zero for the next call with the claim counter) merges the partials:
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
//
// The append instantiation is a whole decode step in one launch: each row's prefix is
// its filled count, the new token's key and value come from the caller's buffers and
// join the final merge in fp32 (score and weight), block 0 of each (row, kv head)
// stores them at the row's next slot once it has streamed its tiles, and the last block
// to arrive on a counter in the meta block advances every row's counters.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

namespace {

constexpr int kWarps = 7;                   // consumer warps
constexpr int kThreads = (kWarps + 1) * 32; // + one producer warp
constexpr int kTile = kWarps * 16;          // 112 slots per stage, 16 per consumer warp
// rows of at most this many tiles: one block, no split merge (the append instantiation's
// split path starts later, without the speculative first tile, so it splits one tile later)
constexpr int kSoloTiles = 4;
constexpr int kSoloTilesAppend = 5;
constexpr int kStages = 4;                  // 4 x 56 KB in flight per SM (bandwidth x loaded latency)
constexpr int kSplitRegs = 5;               // the split merge holds up to 32 x 5 splits' (m, l) in registers
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

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
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

// Per-block abort flag and the limit of its steady-state waits (kTimeoutNs, or the
// testing hook's stall_ns); waits while draining after an abort always use kTimeoutNs.
struct WaitCtl {
  int abort;
  int stall;           // testing hook: steady-state waits wait on `never` instead
  uint64_t limit_ns;
  uint64_t never;      // an mbarrier nothing arrives on
};

// Bounded wait; false when it ran out or the block is aborting.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile WaitCtl* w,
                                          bool honour_abort = true) {
  if (mbar_test_wait(bar, parity)) return true;    // already complete: no flag is read
  if (honour_abort && w->stall) {   // the failure-path test: a wait that nothing ends
    bar = const_cast<uint64_t*>(&w->never);
    parity = 0;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit = honour_abort ? (uint64_t)w->limit_ns : (uint64_t)kTimeoutNs;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (honour_abort && w->abort) return false;
      if (globaltimer() - t0 > limit) {
        w->abort = 1;
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

// ---- warp-level MMA (m16n8k16, 16-bit inputs, fp32 accumulate) -----------------
// ldmatrix reads shared memory that TMA filled: volatile keeps it after the barrier wait.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += A B for A = 16 x 16 (row-major fragment a0..a3, here rows 8..15 are zero: the
// padding of the head dimension) and B = 16 x 8 (fragment b0, b1).
template <typename T>
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float* d, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float* d, uint32_t a0, uint32_t a2, uint32_t b0,
                                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, const __half*) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, const __nv_bfloat16*) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void store_out(__half* p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
// a += w * x, element by element; and four outputs x * inv stored from p on
__device__ __forceinline__ void acc4(float4& a, float w, const float4& x) {
  a.x = fmaf(w, x.x, a.x);
  a.y = fmaf(w, x.y, a.y);
  a.z = fmaf(w, x.z, a.z);
  a.w = fmaf(w, x.w, a.w);
}
template <typename T>
__device__ __forceinline__ void store_out4(T* p, const float4& x, float inv) {
  store_out(p, x.x * inv);
  store_out(p + 1, x.y * inv);
  store_out(p + 2, x.z * inv);
  store_out(p + 3, x.w * inv);
}
__device__ __forceinline__ float load_f(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// K and V tiles are staged as 128-byte-swizzled boxes of 64 dims x kTile slots: 16-byte
// chunk c of slot r sits at chunk c ^ (r & 7) of the slot's 128-byte line, so the 8 row
// addresses of every ldmatrix hit 8 different bank groups.
constexpr uint32_t kHalfBytes = kTile * 128u;                                            // one 64-dim box
template <int D>
__host__ __device__ constexpr uint32_t stage_bytes() { return 2u * (D / 64) * kHalfBytes; }  // K and V
template <int D>
__host__ __device__ constexpr size_t dyn_smem_bytes() { return (size_t)kStages * stage_bytes<D>() + 1024; }

template <typename T, int D, int G, bool kApp>
__global__ void __launch_bounds__(kThreads, 1)
k_decode(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const T* __restrict__ q,
         T* __restrict__ out, int32_t* __restrict__ meta, float* __restrict__ ws, kvc_geom g, float scale_log2,
         float* __restrict__ lse, int fixed_tiles, uint64_t stall_ns, const T* __restrict__ k_new,
         const T* __restrict__ v_new, T* __restrict__ k_store, T* __restrict__ v_store) {
  constexpr int HB = D / 64;         // 64-dim boxes per K (or V) tile
  constexpr int NT = D / 8;          // n-tiles of 8 dims in O
  constexpr uint32_t SB = stage_bytes<D>();
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[kStages], empty[kStages];
  // per-warp partial accumulators [kWarps][G][D]: the stage ring, once every warp is past it
  float (*s_acc)[G][D] = reinterpret_cast<float (*)[G][D]>(dsm);
  __shared__ float s_ml[kWarps][G][2];
  __shared__ float s_inv[G], s_max[G];
  __shared__ int s_last;
  __shared__ float s_snew[G], s_pnew[G];   // append: the new key's score (exp2 domain) and weight
  __shared__ float s_vnew[D];               // append: the new token's value row
  __shared__ WaitCtl s_wc;
  __shared__ int s_tile[kStages];    // tile index held by each stage, -1: no more tiles

  // Blocks launch in linear order onto the SMs; consecutive blocks take different
  // (row, kv head) pairs, so that each pair's splits spread over the whole GPU rather
  // than one region's share of the memory bandwidth.
  const int nsplit = gridDim.x;
  const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int n_pairs = gridDim.y * gridDim.z;
  const int split = lin / n_pairs;
  const int kvh = (lin % n_pairs) % gridDim.y, b = (lin % n_pairs) / gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = lane >> 2;          // head row of this lane in the MMA fragments (real if < G)
  const int quad = lane & 3;         // column pair within the fragments

  // Set-up that touches no global memory runs before the wait for the previous kernel
  // (programmatic dependent launch): the barriers, and the TMA descriptors fetched.
  if (threadIdx.x < kStages) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], kWarps);
  }
  if (threadIdx.x == 0) {
    s_wc.abort = 0;
    s_wc.stall = stall_ns > 0;
    s_wc.limit_ns = stall_ns > 0 ? stall_ns : kTimeoutNs;
    mbar_init(&s_wc.never, 1);
  }
  if (threadIdx.x == kWarps * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_v) : "memory");
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  kvc_pdl_wait();
  kvc_pdl_release();
  // This block's first tile is the same whatever the row's length turns out to be (tile
  // `split`: block 0 of a short row streams tiles 0, 1, ... alone, block s of a split row
  // starts at tile s), and in a LINEAR store its rows do not depend on the meta block:
  // its load is issued before the length is read, so that the two latencies overlap.  A
  // tile past the row's end (or past the store, zero-filled) is loaded and skipped.
  // (Not in the append instantiation, where it measured slower: 5.92 vs 5.68 us a step.)
  const bool spec = !kApp && g.layout == KVC_LINEAR;
  if (spec && warp == kWarps && lane == 0) {
    s_tile[0] = split;                               // published by the arrive below
    mbar_expect_tx(&full[0], SB);
#pragma unroll
    for (int h = 0; h < HB; ++h) {
      tma_load_4d(&tm_k, &full[0], dsm + h * kHalfBytes, 64 * h, kvh, split * kTile, b);
      tma_load_4d(&tm_v, &full[0], dsm + (HB + h) * kHalfBytes, 64 * h, kvh, split * kTile, b);
    }
  }
  // a block that leaves before streaming lets that load land first
  auto leave = [&]() {
    if (spec && warp == kWarps && lane == 0) mbar_wait(&full[0], 0, &s_wc, false);
  };
  // Append-then-attend (k_new set, LINEAR): the row's keys are its `filled` stored slots
  // plus the new token, which this launch also writes to slot `filled`; every block reads
  // its row's length, then the last block to arrive advances every row's meta (reserved
  // chunks, base, filled, kv_len: what kvc_append does) and clears the counter.
  constexpr bool app = kApp;
  constexpr int kNew = kApp ? D / 32 : 1;
  T nk[kNew], nv[kNew], nq[G][kNew];   // append, warp 0: this lane's dims of the new token and queries
  int row0 = 0, len = 0;
  bool row_ok;
  if (app) {
    len = meta[kvc_meta_row(b) + KVC_ROW_FILLED];
    row_ok = len >= 0 && (int64_t)len + 1 <= g.cap;
    if (!row_ok && threadIdx.x == 0 && split == 0 && kvh == 0) atomicOr(meta + KVC_META_ERR, KVC_DEV_OVERFLOW);
    __syncthreads();   // every thread's read of the row's length precedes the arrival below
    if (warp == 0) {
      // Warp 0 alone (the producer warp goes on to issue the first loads, whose latency
      // covers this): arrive, advance every row if this block is the last to arrive, and
      // load the new token's key and value (block 0 of the pair stores them at slot `len`
      // after its stream: no block of this launch reads that slot, and a store there
      // while the first tiles load made the step slower).
      constexpr unsigned kAll = 0xffffffffu;
      int upd = 0;
      if (lane == 0) {
        int prev;
        asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(meta + KVC_META_ARRIVE)
                     : "memory");
        upd = prev == (int)(gridDim.x * gridDim.y * gridDim.z) - 1;
      }
      upd = __shfl_sync(kAll, upd, 0);
      __syncwarp(kAll);   // orders lane 0's acquire before the other lanes' meta writes
      if (upd) {
        for (int bb = lane; bb < g.B; bb += 32) {
          int32_t* m = meta + kvc_meta_row(bb);
          const int f = m[KVC_ROW_FILLED];
          if (f >= 0 && (int64_t)f + 1 <= g.cap) {
            m[KVC_ROW_CHUNKS] += 1;
            m[KVC_ROW_BASE] = f;
            m[KVC_ROW_FILLED] = f + 1;
            m[KVC_ROW_KVLEN] = f + 1;
          }
        }
        __syncwarp(kAll);
        if (lane == 0) meta[KVC_META_ARRIVE] = 0;
      }
      if (row_ok) {   // the new token's key, value and the heads' queries, in flight during the stream
        const int64_t kv_off = ((int64_t)b * g.Hkv + kvh) * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          nk[i] = k_new[kv_off + lane + 32 * i];
          nv[i] = v_new[kv_off + lane + 32 * i];
#pragma unroll
          for (int gg = 0; gg < G; ++gg) nq[gg][i] = q[((int64_t)b * g.H + kvh * G + gg) * D + lane + 32 * i];
        }
      }
    }
  } else {
    row_ok = kvc_row_range(g, b, &row0, &len, meta + KVC_META_ERR);
  }
  if (!row_ok) {
    leave();
    return;
  }

  // Tiles of kTile slots of this row: block `split` takes tiles split, split + nsplit, ...
  // for its first kStages tiles, then claims tiles kStages * nsplit, ... one at a time
  // from the (row, kv head) counter, so blocks that stream faster take more tiles.
  const int n_row_tiles = (len + kTile - 1) / kTile;
  // A short row is streamed by block 0 of its (row, kv head) alone, which writes the
  // output directly: for a few tiles the split merge (partials, ticket, last-block
  // merge) costs more than one block streaming them.  Uniform per block.
  const bool solo = n_row_tiles <= (kApp ? kSoloTilesAppend : kSoloTiles);
  if (solo && split != 0) {
    leave();
    return;
  }
  const int pairs = g.B * g.Hkv;
  const int pair = b * g.Hkv + kvh;
  float* ws_o = ws;                                              // [pairs][nsplit][G][D]
  float* ws_ml = ws + (int64_t)pairs * nsplit * G * D;           // [pairs][nsplit][G][2]
  int* tickets = reinterpret_cast<int*>(ws_ml + (int64_t)pairs * nsplit * G * 2);  // [pairs]
  int* claims = tickets + pairs;                                 // [pairs]

  volatile WaitCtl* abort = &s_wc;

  if (warp == kWarps) {
    // ---------------- producer: TMA tiles of K and V into the stage ring ----------------
    if (lane == 0) {
      const int kv_batch = g.layout == KVC_PACKED ? 0 : b;
      int issued = spec ? 1 : 0;
      // tile t of this block: static for t < kStages, else claimed.  Claims are issued two
      // tiles ahead, so that their round trips overlap the streaming of two tiles.
      auto claim_for = [&](int t) {   // fixed_tiles: tile t is split + t * nsplit throughout
        if (solo) return t;
        return t < kStages || fixed_tiles ? split + t * nsplit : kStages * nsplit + atomicAdd(claims + pair, 1);
      };
      auto step = [&](int t, int tile) {
        const int st = t % kStages;
        if (t == 0 && spec) return true;                 // issued before the length was read
        if (t >= kStages && !mbar_wait(&empty[st], ((t / kStages) - 1) & 1, abort)) return false;
        if (tile >= n_row_tiles) {                       // no more tiles: tell the consumers
          s_tile[st] = -1;
          mbar_arrive(&full[st]);
          return false;
        }
        s_tile[st] = tile;                               // published by the arrive below
        mbar_expect_tx(&full[st], SB);
        uint8_t* dst = dsm + st * SB;
        const int row = row0 + tile * kTile;
#pragma unroll
        for (int h = 0; h < HB; ++h) {
          tma_load_4d(&tm_k, &full[st], dst + h * kHalfBytes, 64 * h, kvh, row, kv_batch);
          tma_load_4d(&tm_v, &full[st], dst + (HB + h) * kHalfBytes, 64 * h, kvh, row, kv_batch);
        }
        issued = t + 1;
        return true;
      };
      static_assert(kStages >= 2, "the first two tiles are static");
      int ca = claim_for(0), cb = claim_for(1);
      for (int t = 0;; t += 2) {                         // claims are monotonic: none is skipped
        if (!step(t, ca)) break;
        ca = claim_for(t + 2);
        if (!step(t + 1, cb)) break;
        cb = claim_for(t + 3);
      }
      if (abort->abort) {   // let every load issued here land before the block releases its shared memory
        for (int t = max(0, issued - kStages); t < issued; ++t)
          mbar_wait(&full[t % kStages], (t / kStages) & 1, abort, false);
      }
    }
  }

  // Per warp and tile: S = Q K^T on this warp's 16 slots (M = heads padded to 16, N = 8
  // slots per MMA, K = 16 dims per MMA), online softmax per head row, O += P V (M = heads,
  // N = 8 dims, K = the 16 slots).  The S fragment of two slot n-tiles is the P fragment
  // of the PV MMA, so P never leaves registers.  Lane: head row hq, slots/dims 2 quad, +1.
  uint32_t qa[D / 16][2];            // A fragments of Q (unscaled; rows 8..15 are zero)
  float o[NT][4];                    // O fragments: rows hq (real heads) and hq + 8 (padding)
  float m = -INFINITY, l = 0.f;      // running max (exp2 domain) and sum of this lane's head row
  if (warp < kWarps) {
    const T* qp = q + ((int64_t)b * g.H + kvh * G + (hq < G ? hq : 0)) * D + 2 * quad;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = hq < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk)) : 0u;
      qa[kk][1] = hq < G ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kk + 8)) : 0u;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    const int r0 = warp * 16;                              // this warp's slots of every tile
    for (int t = 0;; ++t) {
      const int st = t % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (t / kStages) & 1, abort))) break;
      const int tile = s_tile[st];
      if (tile < 0) break;
      const uint32_t kbase = smem_u32(dsm + st * SB);
      const uint32_t vbase = kbase + HB * kHalfBytes;
      const int first = tile * kTile + r0;                 // row index of slot r0
      if (first < len) {
        if (first + 16 > len) {
          // slots past the valid range may hold anything (NaN included): zero their V rows
          // so that P = 0 there contributes exactly nothing
          uint8_t* vrow = dsm + st * SB + HB * kHalfBytes;
          for (int e = lane; e < 16 * HB * 8; e += 32) {
            const int r = r0 + e / (HB * 8), h = (e / 8) % HB, c = e % 8;
            if (tile * kTile + r >= len)
              *reinterpret_cast<uint4*>(vrow + h * kHalfBytes + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // before TMA reuses the stage
          __syncwarp();
        }
        // S: ldmatrix x4 = (slots r0..7 | r0+8..15) x (dims 16kk..+7 | +8..+15)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int j = lane >> 3, i = lane & 7;
          const int slot = r0 + (j >> 1) * 8 + i;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int chunk = (kk & 3) * 2 + (j & 1);
            uint32_t bk[4];
            ldsm_x4(kbase + (kk >> 2) * kHalfBytes + slot * 128 + ((chunk ^ (slot & 7)) << 4), bk);
            mma16816<T>(sc[0], qa[kk][0], qa[kk][1], bk[0], bk[1]);
            mma16816<T>(sc[1], qa[kk][0], qa[kk][1], bk[2], bk[3]);
          }
        }
        // online softmax of head row hq over the warp's 16 slots
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int sl = first + (e >> 1) * 8 + 2 * quad + (e & 1);
          x[e] = sl < len ? sc[e >> 1][e & 1] * scale_log2 : -INFINITY;
        }
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (mx > m) {                                      // the running max grows
          const float alpha = ex2(m - mx);                 // 0 on the first tile (m = -inf)
          m = mx;
          l *= alpha;
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            o[n][0] *= alpha;
            o[n][1] *= alpha;
          }
        }
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pr[e] = ex2(x[e] - m);
          l += pr[e];
        }
        const uint32_t pa0 = pack2(pr[0], pr[1], (const T*)nullptr);   // slots 2 quad, +1
        const uint32_t pa2 = pack2(pr[2], pr[3], (const T*)nullptr);   // slots 8 + 2 quad, +1
        // O += P V: ldmatrix.trans x4 = (slots r0..7 | r0+8..15) x (dims 8n..+7 | 8n+8..+15)
        {
          const int j = lane >> 3, i = lane & 7;
          const int slot = r0 + (j & 1) * 8 + i;
#pragma unroll
          for (int n = 0; n < NT; n += 2) {
            const int chunk = (n & 7) + (j >> 1);
            uint32_t bv[4];
            ldsm_x4_t(vbase + (n >> 3) * kHalfBytes + slot * 128 + ((chunk ^ (slot & 7)) << 4), bv);
            mma16816<T>(o[n], pa0, pa2, bv[0], bv[1]);
            mma16816<T>(o[n + 1], pa0, pa2, bv[2], bv[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);           // this warp is done with the stage
    }
    // the 4 lanes of a quad summed different slots of the same head row
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
  }
  if (app && warp == 0) {   // the new key's score per head (exp2 domain) and its value row
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc = fmaf(load_f(&nq[gg][i]), load_f(&nk[i]), acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) s_snew[gg] = acc * scale_log2;
    }
#pragma unroll
    for (int i = 0; i < D / 32; ++i) s_vnew[lane + 32 * i] = load_f(&nv[i]);
  }
  __syncthreads();                                  // every warp (and every load) is done with the ring
  if (warp < kWarps && hq < G) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      s_acc[warp][hq][8 * n + 2 * quad] = o[n][0];
      s_acc[warp][hq][8 * n + 2 * quad + 1] = o[n][1];
    }
    if (quad == 0) {
      s_ml[warp][hq][0] = m;
      s_ml[warp][hq][1] = l;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_wc.abort) atomicOr(meta + KVC_META_ERR, KVC_DEV_TIMEOUT);
  if (app && split == 0 && warp == 0) {   // the new token's K and V rows, at slot len
    T* kd = k_store + (((int64_t)b * g.cap + len) * g.Hkv + kvh) * D;
    T* vd = v_store + (((int64_t)b * g.cap + len) * g.Hkv + kvh) * D;
#pragma unroll
    for (int i = 0; i < kNew; ++i) {
      kd[lane + 32 * i] = nk[i];
      vd[lane + 32 * i] = nv[i];
    }
  }

  // ---- this block's partial: merge the warps ---------------------------------
  if (solo) {   // the whole row: normalise and write the output
    if (threadIdx.x < G) {
      const int gg = threadIdx.x;
      float M = -INFINITY, L = 0.f;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][gg][0]);
      for (int w = 0; w < kWarps; ++w) {
        const float mw = s_ml[w][gg][0];
        if (mw != -INFINITY) L = fmaf(ex2(mw - M), s_ml[w][gg][1], L);
      }
      if (app) {   // the new key joins with weight 2^(s - M)
        const float sn = s_snew[gg], M2 = fmaxf(M, sn);
        L = (M == -INFINITY ? 0.f : L * ex2(M - M2)) + ex2(sn - M2);
        M = M2;
        s_pnew[gg] = ex2(sn - M);
      }
      s_max[gg] = M;
      s_inv[gg] = 1.f / L;
      if (lse != nullptr) lse[(int64_t)b * g.H + kvh * G + gg] = (M + log2f(L)) * 0.6931471805599453f;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < G * D / 4; v += blockDim.x) {   // 4 outputs of one head each
      const int gg = (4 * v) / D, d = 4 * v - gg * D;
      const float M = s_max[gg];
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = s_ml[w][gg][0];
        if (mw != -INFINITY) acc4(a, ex2(mw - M), *reinterpret_cast<const float4*>(&s_acc[w][gg][d]));
      }
      if (app) acc4(a, s_pnew[gg], make_float4(s_vnew[d], s_vnew[d + 1], s_vnew[d + 2], s_vnew[d + 3]));
      store_out4(out + ((int64_t)b * g.H + kvh * G + gg) * D + d, a, s_inv[gg]);
    }
    return;
  }
  for (int v = threadIdx.x; v < G * D / 4; v += blockDim.x) {     // 4 outputs of one head each
    const int gg = (4 * v) / D, d = 4 * v - gg * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][gg][0]);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = s_ml[w][gg][0];
      if (mw != -INFINITY) acc4(a, ex2(mw - M), *reinterpret_cast<const float4*>(&s_acc[w][gg][d]));
    }
    reinterpret_cast<float4*>(ws_o + ((int64_t)pair * nsplit + split) * G * D)[v] = a;
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
  // The block's partial stores precede thread 0's acq_rel ticket (block barrier, then a
  // release that is cumulative over them); the last block's loads follow its acquire.
  __syncthreads();
  if (threadIdx.x == 0) {
    int prev;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(prev) : "l"(tickets + pair) : "memory");
    s_last = prev == nsplit - 1;
  }
  __syncthreads();
  if (!s_last) return;

  // ---- merge the splits (last block of this (b, kv head)) -------------------
  // Thread t owns the 16-byte output groups v = t + i * blockDim.x (outputs 4v .. 4v + 3,
  // one head) and loads their first kPre split partials at once, 16 bytes a load (one L2
  // round trip, in flight while the weights are formed); the weights 2^(m_s - M) of each
  // head go to shared memory (the stage ring is free now), then
  // O = sum_s w_s O_s / sum_s w_s l_s.
  constexpr int kVec = G * D / 4;                                  // 16-byte groups of outputs
  constexpr int kOut4 = (kVec + kThreads - 1) / kThreads;         // groups per thread
  constexpr int kPre = 24 / kOut4;                                 // splits prefetched per group
  const int used = min(nsplit, n_row_tiles);                     // blocks past the tile count took none
  const float4* ws_pair = reinterpret_cast<const float4*>(ws_o + (int64_t)pair * nsplit * G * D);
  float4 pre[kOut4][kPre];
#pragma unroll
  for (int i = 0; i < kOut4; ++i) {
    const int v = threadIdx.x + i * kThreads;
#pragma unroll
    for (int k = 0; k < kPre; ++k)
      pre[i][k] = (v < kVec && k < used) ? __ldcg(ws_pair + (int64_t)k * kVec + v) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // One warp per head: lane s takes split s's (m_s, l_s) straight into registers (up to
  // kSplitRegs splits), forms M and the weights, and leaves them in shared memory for
  // the output groups: one barrier between the loads and the outputs.
  float* sw = reinterpret_cast<float*>(dsm);                     // [G][used] weights
  for (int gg = warp; gg < G; gg += kWarps + 1) {
    float mr[kSplitRegs], lr[kSplitRegs];
#pragma unroll
    for (int j = 0; j < kSplitRegs; ++j) {
      const int sp = lane + 32 * j;
      mr[j] = -INFINITY;
      lr[j] = 0.f;
      if (sp < used) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(ws_ml + (((int64_t)pair * nsplit + sp) * G + gg) * 2));
        mr[j] = ml.x;
        lr[j] = ml.y;
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < kSplitRegs; ++j) M = fmaxf(M, mr[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (app) M = fmaxf(M, s_snew[gg]);
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kSplitRegs; ++j) {
      const int sp = lane + 32 * j;
      if (sp < used) {
        const float wgt = mr[j] == -INFINITY ? 0.f : ex2(mr[j] - M);
        sw[gg * used + sp] = wgt;
        L = fmaf(wgt, lr[j], L);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) {
      if (app) {   // the new key joins with weight 2^(s - M)
        s_pnew[gg] = ex2(s_snew[gg] - M);
        L += s_pnew[gg];
      }
      s_inv[gg] = 1.f / L;
      if (lse != nullptr) lse[(int64_t)b * g.H + kvh * G + gg] = (M + log2f(L)) * 0.6931471805599453f;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kOut4; ++i) {
    const int v = threadIdx.x + i * kThreads;
    if (v >= kVec) break;
    const int gg = (4 * v) / D, d = 4 * v - gg * D;
    const float* wrow = sw + gg * used;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kPre; ++k)
      if (k < used) acc4(o, wrow[k], pre[i][k]);
    for (int k = kPre; k < used; ++k) acc4(o, wrow[k], __ldcg(ws_pair + (int64_t)k * kVec + v));
    if (app) acc4(o, s_pnew[gg], make_float4(s_vnew[d], s_vnew[d + 1], s_vnew[d + 2], s_vnew[d + 3]));
    store_out4(out + ((int64_t)b * g.H + kvh * G + gg) * D + d, o, s_inv[gg]);
  }
  if (threadIdx.x == 0) {           // every block of the pair is past both counters
    tickets[pair] = 0;
    claims[pair] = 0;
  }
}

// The new token of an append-then-attend decode ([B, 1, Hkv, D] each), or none.
struct DecAppend {
  const void* k = nullptr;
  const void* v = nullptr;
};

template <typename T, int D, int G>
cudaError_t launch_dg(kvc_cache* c, const void* q, void* out, float* lse, int fixed, cudaStream_t s, bool prepare,
                      const DecAppend& ap) {
  constexpr size_t smem = dyn_smem_bytes<D>();
  if (prepare) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_decode<T, D, G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_decode<T, D, G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  }
  const kvc_config& cfg = c->cfg;
  if (c->dec_splits > 32 * kSplitRegs) return cudaErrorInvalidValue;   // the merge's register budget
  kvc_geom g{cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim, c->cap, cfg.layout, c->lens};
  dim3 grid(c->dec_splits, cfg.kv_heads, cfg.batch);
  const float sl2 = c->scale * 1.4426950408889634f;
  if (ap.k == nullptr)
    return kvc_launch_pdl(k_decode<T, D, G, false>, grid, dim3(kThreads), smem, s, c->tm_dk, c->tm_dv, (const T*)q,
                          (T*)out, c->meta, (float*)c->ws, g, sl2, lse, fixed, c->debug_stall_ns, (const T*)nullptr,
                          (const T*)nullptr, (T*)c->k, (T*)c->v);
  return kvc_launch_pdl(k_decode<T, D, G, true>, grid, dim3(kThreads), smem, s, c->tm_dk, c->tm_dv, (const T*)q,
                        (T*)out, c->meta, (float*)c->ws, g, sl2, lse, fixed, c->debug_stall_ns, (const T*)ap.k,
                        (const T*)ap.v, (T*)c->k, (T*)c->v);
}

template <typename T, int D>
cudaError_t launch_d(kvc_cache* c, const void* q, void* out, float* lse, int fixed, cudaStream_t s, bool prepare,
                     const DecAppend& ap) {
  switch (c->cfg.heads / c->cfg.kv_heads) {
    case 1: return launch_dg<T, D, 1>(c, q, out, lse, fixed, s, prepare, ap);
    case 2: return launch_dg<T, D, 2>(c, q, out, lse, fixed, s, prepare, ap);
    case 4: return launch_dg<T, D, 4>(c, q, out, lse, fixed, s, prepare, ap);
    default: return launch_dg<T, D, 8>(c, q, out, lse, fixed, s, prepare, ap);
  }
}

template <typename T>
cudaError_t launch_t(kvc_cache* c, const void* q, void* out, float* lse, int fixed, cudaStream_t s, bool prepare,
                     const DecAppend& ap = DecAppend()) {
  return c->cfg.head_dim == 64 ? launch_d<T, 64>(c, q, out, lse, fixed, s, prepare, ap)
                               : launch_d<T, 128>(c, q, out, lse, fixed, s, prepare, ap);
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
  e = ti == 0 ? launch_t<__half>(c, nullptr, nullptr, nullptr, 0, 0, true)
              : launch_t<__nv_bfloat16>(c, nullptr, nullptr, nullptr, 0, 0, true);
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
  return pairs * splits * G * (cfg.head_dim + 2) * 4 + pairs * 8;   // partials, tickets, tile claims
}

cudaError_t kvc_prepare_decode(kvc_cache* c) { return prepare_once(c); }

bool kvc_make_decode_maps(kvc_cache* c) {
  const kvc_config& g = c->cfg;
  const uint64_t batches = g.layout == KVC_PACKED ? 1 : (uint64_t)g.batch;
  const uint64_t cap = (uint64_t)c->cap;
  return kvc_make_tile_map(&c->tm_dk, g.dtype, c->k, g.head_dim, g.kv_heads, cap, batches, kTile, KVC_BOX_SW128) &&
         kvc_make_tile_map(&c->tm_dv, g.dtype, c->v, g.head_dim, g.kv_heads, cap, batches, kTile, KVC_BOX_SW128);
}

cudaError_t kvc_launch_decode(kvc_cache* c, const void* q, void* out, float* lse, bool fixed_tiles,
                              cudaStream_t s) {
  const cudaError_t e = prepare_once(c);
  if (e != cudaSuccess) return e;
  const int fixed = fixed_tiles ? 1 : 0;
  return c->cfg.dtype == KVC_F16 ? launch_t<__half>(c, q, out, lse, fixed, s, false)
                                 : launch_t<__nv_bfloat16>(c, q, out, lse, fixed, s, false);
}

cudaError_t kvc_launch_decode_append(kvc_cache* c, const void* k_new, const void* v_new, const void* q, void* out,
                                     cudaStream_t s) {
  const cudaError_t e = prepare_once(c);
  if (e != cudaSuccess) return e;
  DecAppend ap;
  ap.k = k_new;
  ap.v = v_new;
  return c->cfg.dtype == KVC_F16 ? launch_t<__half>(c, q, out, nullptr, 0, s, false, ap)
                                 : launch_t<__nv_bfloat16>(c, q, out, nullptr, 0, s, false, ap);
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
  c.lens = meta;
  c.ws = scratch;
  c.dec_splits = splits;
  if (!kvc_make_decode_maps(&c)) return KVC_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the tickets sit after the partials; an earlier call with another shape may have
  // left partial data there
  const size_t pairs = (size_t)cfg->batch * cfg->kv_heads;
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - pairs * 8), 0, pairs * 8, s) != cudaSuccess)
    return KVC_ERR_CUDA;
  return kvc_launch_decode(&c, q, out, nullptr, false, s) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}
