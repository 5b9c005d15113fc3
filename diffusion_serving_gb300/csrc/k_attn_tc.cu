// Tensor-core chunk attention for bf16 / fp16, D = 128 (sm_103a: tcgen05 + TMEM + TMA).
// Two kernels share the helpers below: k_attn_tc (a pair of query tiles per item, for
// stores of at most kShortKv slots per row) and k_attn_1q (one query tile per item with
// S triple-buffered in TMEM, for longer stores); the launcher picks by shape.
//
// Computes, for every query row of a chunk, softmax(scale * q K^T) V over the row's
// valid slots in physical order: [0, kv_len) of a LINEAR or CIRCULAR store (the
// circular sink+window ring is attended as stored, since permuting K and V rows
// together leaves unmasked attention unchanged — flashdreams issue "add an opt-in
// circular KV policy for streaming attention", "proposed boundary"), or
// [cu_b, cu_{b+1}) of a PACKED store (TensorRT-LLM PR "FA4 variable-length
// cross-attention", Description).  Only the active prefix is read (fish-speech PR
// "pass only active KV cache prefix to SDPA", "Change"); with KVC_CAUSAL the query
// at absolute position kv_len - n_q + i sees slots <= that position (same section).
//
// The pair kernel, k_attn_tc (the one-tile kernel is described above its definition):
// work item = two 128-row query tiles (A and B) of one (batch row, q head), sharing
// every K/V tile it loads.  The kernel is persistent: one CTA per SM walks the items.
// Warp roles (384 threads):
//   warps 0, 3  TMA producers (warp 0 the item's Q tiles and K, warp 3 V): tiles of 128
//               slots into two-stage rings (128B-swizzled boxes of 64 dims x 128 slots).
//   warps 1, 2  MMA issuers, one per query tile (warp 1 also owns TMEM): S = Q K^T
//               (A, B from shared memory) and O += P V (P from TMEM, V from shared
//               memory), fp32 accumulators in TMEM.
//   warps 4-7   softmax of tile A, one query row per thread: S row from TMEM, online
//               max / exp2 / sum, P written back to TMEM over S, O rescaled in TMEM
//               when the row max grows by more than 2^8; at the end O / l goes to
//               global memory through 64-byte-swizzled shared staging and TMA stores.
//               A short last tile (no causal mask) skips its 32-column chunks past the
//               valid slots; with the causal mask, only a tile that crosses the
//               diagonal for some row of the warp is masked (a warp vote per tile).
//   warps 8-11  the same for tile B.
// TMEM columns: S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512); P_X occupies the
// first 64 columns of S_X as packed 16-bit pairs.
//
// MMA order per K/V tile j: PV_A(j), QK_A(j+1) from warp 1 and PV_B(j), QK_B(j+1) from
// warp 2, with B's PV(j) issued after A's and A's PV(j+1) after B's PV(j) (the order of
// a single issuer, at half-group granularity, so that the tiles' softmaxes alternate).
// A single thread issues MMAs at most every ~100 cycles while the tensor pipe retires
// one per 64, so two issuing warps overlap one tile's QK with the other's PV.  The
// commit that signals "S_X(j+1) ready" also covers PV_X(j) (same thread, in order), so
// when the softmax warps see S_X(j+1) the O_X accumulator is stable and may be rescaled.
//
// Every mbarrier wait is bounded (0.5 s of %globaltimer); on expiry the kernel records
// KVC_DEV_TIMEOUT, drains its own TMA loads and MMAs, frees TMEM and returns, and CTAs
// that start after the error word carries KVC_DEV_TIMEOUT return at once.
#include "kvc_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

namespace {

constexpr int kD = 128;
constexpr int kBM = 128;            // query rows per tile
constexpr int kBN = 128;            // slots per K/V tile
constexpr int kStages = 2;
constexpr int kThreads = 384;
constexpr int kShortKv = 1024;      // stores of at most this many slots per row: the query-tile-pair kernel
constexpr uint32_t kBoxBytes = 64 * 2 * 128;         // 64 dims x 128 rows, 16-bit
constexpr uint32_t kTileBytes = 2 * kBoxBytes;       // 128 dims
constexpr uint32_t kStageBytes = 32 * 32 * 2;        // 32 rows x 32 dims, 16-bit
constexpr uint64_t kTimeoutNs = 500000000ull;   // 0.5 s; a healthy wait is microseconds
constexpr float kRescaleThreshold = 8.0f;            // log2 units
constexpr float kRescaleSum = 256.0f;                // 2^kRescaleThreshold

// Per-CTA abort flag and the limit of its steady-state waits (kTimeoutNs, or the testing
// hook's stall_ns); waits while draining after an abort always use kTimeoutNs.
struct WaitCtl {
  int abort;
  int stall;           // testing hook: steady-state waits wait on `never` instead
  uint64_t limit_ns;
  uint64_t never;      // an mbarrier nothing arrives on
};

struct Smem {
  // 1024-byte aligned tiles (128B swizzle atoms)
  uint8_t q[2][kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  // output staging: per softmax warp two 32-row x 32-column buffers (64-byte swizzle),
  // written to global memory by TMA stores
  uint8_t o_stage[8][2][kStageBytes];
  uint64_t q_full, q_free;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t v_ready[kStages];   // V tile with its invalid rows zeroed (warp 1 -> warp 2)
  uint64_t tok[2];             // issue order: tok[t] = issuer t has issued its PV of tile j
  uint64_t s_full[2], p_ready[2], o_done[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  WaitCtl wc;
};

static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory above the 227 KB a block may opt into");
static_assert(offsetof(Smem, o_stage) % 1024 == 0, "staging buffers must keep the swizzle phase of their address");

// ---- PTX wrappers ----------------------------------------------------------
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

// Bounded wait for the phase with the given parity.  Returns false when the CTA is
// aborting (another role gave up) or when this wait ran out of time (then it starts
// the abort itself).  `honour_abort` = false is used while draining.
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

// Bulk tensor store of one box from shared memory; completion tracked by bulk groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2,
                                             int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(map),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until every committed bulk group has completed its writes
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulate, A/B 16-bit (fmt 0 fp16, 1 bf16),
// A K-major, B K-major or MN-major, M = 128, N = 128.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t fmt, uint32_t b_mn_major) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn_major << 16) | ((uint32_t)(kBN >> 3) << 17) |
         ((uint32_t)(kBM >> 4) << 24);
}

// Shared-memory matrix descriptor (128-byte swizzle, sm_100 descriptor version) as its
// two 32-bit words: start address >> 4 in bits 0-13, leading-byte offset >> 4 in 16-29,
// stride-byte offset >> 4 in 32-45, bit 46 set, layout 2 (128-byte swizzle) in 61-63.
// The K steps of one MMA sequence differ only in the start address, so a sequence builds
// the words once and adds each step's offset >> 4 to the low word: one 32-bit add per
// step instead of rebuilding the 64-bit descriptor.  The address field is
// (addr >> 4) & 0x3FFF; shared addresses are below 227 KB (< 14,528 in that unit) and a
// step offset is at most 16,480 bytes (1,030), so the add never carries out of the field.
struct SDesc {
  uint32_t lo, hi;
};
__device__ __forceinline__ SDesc sdesc2(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return {((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16),
          ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29)};
}
// kind::f16 MMA, A and B from shared memory: descriptors a and b advanced by a_off /
// b_off bytes.
__device__ __forceinline__ void mma_ss2(uint32_t d, SDesc a, uint32_t a_off, SDesc b, uint32_t b_off,
                                        uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d),
      "r"(a.lo + (a_off >> 4)), "r"(a.hi), "r"(b.lo + (b_off >> 4)), "r"(b.hi), "r"(idesc), "r"(acc)
      : "memory");
}
// kind::f16 MMA, A from TMEM, B from shared memory advanced by b_off bytes.
__device__ __forceinline__ void mma_ts2(uint32_t d, uint32_t a_tmem, SDesc b, uint32_t b_off, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(b.lo + (b_off >> 4)), "r"(b.hi), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

#define KVC_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
#define KVC_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), \
                  "r"(r[i + 7])

// 32 TMEM lanes (one per thread of the warp) x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : KVC_R8(0), KVC_R8(8), KVC_R8(16), KVC_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      KVC_W8(0), KVC_W8(8), KVC_W8(16), KVC_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Ties 32 registers filled by tmem_ld32 to the preceding wait, so that no use of them
// is scheduled before the asynchronous load has completed.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
               "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
               "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
               "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      KVC_W8(0), KVC_W8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Per-warpgroup register split (all four warps of a warpgroup execute it): the pair
// kernel launches 384 threads x 168 registers = 64,512; warps 0-3 (TMA producers and MMA
// issuers) give theirs down to 88 and the two softmax warpgroups take 208 each:
// 128 x 88 + 256 x 208 = 64,512, the launch's total, so every increase is served.  The
// launcher checks that the compiled kernel does launch with 168 registers per thread
// (an increase beyond the launch's total would never be served).
template <uint32_t kRegs> __device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs> __device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
constexpr uint32_t kRegsLaunch = 168, kRegsCtl = 88, kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split above the launch's total");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (kBf16)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Row max of the 128 scores a thread holds, over columns < valid when kMask (eight
// independent chains of 3-input maxima so that the reduction is not one long
// dependency).
template <bool kMask, int kChunks>
__device__ __forceinline__ float row_max(const uint32_t* sr, int valid) {
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32 * kChunks; i += 2) {
    float x0 = __uint_as_float(sr[i]), x1 = __uint_as_float(sr[i + 1]);
    if (kMask) {
      x0 = i < valid ? x0 : -INFINITY;
      x1 = i + 1 < valid ? x1 : -INFINITY;
    }
    mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], x0, x1);
  }
  return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
}

// p = 2^(s * c - m) for the first 32 * kChunks columns (0 past `valid` when kMask),
// packed as 16-bit pairs over the first 64 TMEM columns of the row's S; with kZeroRest
// the P of the chunks past kChunks is stored as 0 (for a PV MMA that reads all 128).
// Returns the row sum of p.  Pairs of columns go through the packed fp32x2 FMA / add.
template <bool kBf16, bool kMask, int kChunks, bool kZeroRest = true>
__device__ __forceinline__ float exp_pack_store(const uint32_t* sr, int valid, float c, float m_use, uint32_t s_addr) {
  const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_use, -m_use);
  float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if (kChunks < 4 && kZeroRest) {
    uint32_t zero[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) zero[i] = 0u;
#pragma unroll
    for (int q4 = kChunks; q4 < 4; ++q4) tmem_st16(s_addr + q4 * 16, zero);
  }
#pragma unroll
  for (int q4 = 0; q4 < kChunks; ++q4) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c0 = q4 * 32 + 2 * i;
      const float2 t = __ffma2_rn(make_float2(__uint_as_float(sr[c0]), __uint_as_float(sr[c0 + 1])), c2, nm2);
      float x0 = ex2(t.x), x1 = ex2(t.y);
      if (kMask) {
        x0 = c0 < valid ? x0 : 0.f;
        x1 = c0 + 1 < valid ? x1 : 0.f;
      }
      sum[i & 1] = __fadd2_rn(sum[i & 1], make_float2(x0, x1));
      pk[i] = pack2<kBf16>(x0, x1);
    }
    tmem_st16(s_addr + q4 * 16, pk);
  }
  return (sum[0].x + sum[0].y) + (sum[1].x + sum[1].y);
}

struct TcParams {
  kvc_geom g;
  int n_q;
  int causal;
  float scale_log2;
  float* lse;        // optional [B, n_q, H] natural-log log-sum-exp of each row's scaled scores
  uint64_t stall_ns; // testing hook: > 0 makes steady-state waits wait this long on a barrier
                     // nothing arrives on (then the CTA aborts); 0 in normal use
};

// Work item = one pair of 128-row query tiles (A, B) of one (batch row, q head), in the
// order pair-fastest, then head, then row.  The same geometry is derived independently
// by every role from the item index and the meta block.
struct Item {
  int b, h, kvh, row_a, row0, kv_batch, qpos0, kv_end, n_tiles;
};

// Row range of the last batch row looked up (consecutive items of a CTA mostly share
// it), so that the meta block is read once per row and role rather than once per item.
struct RowCache {
  int b = -1, row0 = 0, len = 0;
  bool ok = false;
};

__device__ __forceinline__ bool item_geom(int item, int pairs, const TcParams& p, int32_t* meta, RowCache& rc,
                                          Item* it) {
  const kvc_geom& g = p.g;
  const int pair = item % pairs, bh = item / pairs;
  it->h = bh % g.H;
  it->b = bh / g.H;
  it->kvh = it->h / (g.H / g.Hkv);
  it->row_a = pair * 2 * kBM;
  if (it->b != rc.b) {
    rc.b = it->b;
    rc.ok = kvc_row_range(g, it->b, &rc.row0, &rc.len, meta + KVC_META_ERR);
  }
  if (!rc.ok) return false;
  const int len = rc.len;
  it->row0 = rc.row0;
  it->kv_batch = g.layout == KVC_PACKED ? 0 : it->b;
  it->qpos0 = len - p.n_q;                             // absolute position of query 0 (causal)
  it->kv_end = len;
  if (p.causal) {
    const int last_row = min(it->row_a + 2 * kBM, p.n_q) - 1;
    it->kv_end = max(1, min(len, it->qpos0 + last_row + 1));
  }
  it->n_tiles = (it->kv_end + kBN - 1) / kBN;
  return true;
}

// ---- the kernel --------------------------------------------------------------
// Persistent: one CTA per SM walks the work items item = blockIdx.x, + gridDim.x, ...
// Barrier phases continue across items: K/V stages, S-ready and P-ready barriers count
// K/V tiles over the CTA's whole run, the Q and O barriers count items.  The next
// item's Q tiles load as soon as the current item's last QK MMA has completed, and its
// first MMAs run while the softmax warps finish the current item's epilogue.
template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
          int32_t* __restrict__ meta, TcParams p) {
  kvc_pdl_wait();   // launched as a programmatic dependent: nothing is read before this
  kvc_pdl_release();
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const kvc_geom& g = p.g;
  const int pairs = (p.n_q + 2 * kBM - 1) / (2 * kBM);
  const int n_items = g.B * g.H * pairs;

  // a CTA that starts after another one gave up on a wait returns at once (one read,
  // shared, so that every thread takes the same branch)
  if (threadIdx.x == 0) {
    sm.wc.abort = (*reinterpret_cast<volatile int32_t*>(meta + KVC_META_ERR) & KVC_DEV_TIMEOUT) ? 1 : 0;
    sm.wc.limit_ns = p.stall_ns > 0 ? p.stall_ns : kTimeoutNs;
    sm.wc.stall = p.stall_ns > 0;
  }
  __syncthreads();
  if (sm.wc.abort) return;
  volatile WaitCtl* abort = &sm.wc;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, 2);   // both issuers' last QK of the item
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 2);   // QK of both query tiles
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 2);   // PV of both query tiles
      mbar_init(&sm.v_ready[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_ready[t], kBM / 32);   // one arrival per softmax warp
      mbar_init(&sm.o_done[t], 1);
    }
    mbar_init(&sm.tok[0], 1);
    mbar_init(&sm.tok[1], 1);
    mbar_init(&sm.drain[0], 1);
    mbar_init(&sm.drain[1], 1);
    mbar_init(&sm.wc.never, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // the register split comes first in each role's code (so the compiler sizes each role's
  // code by its own share)
  if (warp < 4) {
   regs_dec<kRegsCtl>();
   if (warp == 0 || warp == 3) {
    // ---------------- TMA producers: warp 0 Q and K, warp 3 V ----------------
    // (two threads, so that a K load never queues behind a V load waiting for a PV)
    if (lane == 0) {
      const bool kq = warp == 0;
      int T = 0, n_items_done = 0;           // K/V tiles and items issued so far
      RowCache rc;
      int issued = 0, q_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        Item I;
        if (!item_geom(item, pairs, p, meta, rc, &I)) continue;
        if (kq) {
          // the previous item's Q tiles are free once its last QK MMA completed
          if (n_items_done > 0 && !mbar_wait(&sm.q_free, (n_items_done - 1) & 1, abort)) break;
          mbar_expect_tx(&sm.q_full, 2 * kTileBytes);
          for (int t = 0; t < 2; ++t)
            for (int half = 0; half < 2; ++half)
              tma_load_4d(&tm_q, &sm.q_full, sm.q[t] + half * kBoxBytes, half * 64, I.h, I.row_a + t * kBM, I.b);
          q_issued = n_items_done + 1;
        }
        const CUtensorMap* tm = kq ? &tm_k : &tm_v;
        for (int j = 0; j < I.n_tiles; ++j) {
          const int Tj = T + j, s = Tj % kStages, u = Tj / kStages;
          uint64_t* empty = kq ? &sm.k_empty[s] : &sm.v_empty[s];
          uint64_t* full = kq ? &sm.k_full[s] : &sm.v_full[s];
          uint8_t* dst = kq ? sm.k[s] : sm.v[s];
          if (Tj >= kStages && !mbar_wait(empty, (u - 1) & 1, abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full, kTileBytes);
          for (int half = 0; half < 2; ++half)
            tma_load_4d(tm, full, dst + half * kBoxBytes, half * 64, I.kvh, I.row0 + j * kBN, I.kv_batch);
          issued = Tj + 1;
        }
        T += I.n_tiles;
        ++n_items_done;
      }
      if (abort->abort) {
        // drain: every load this thread issued lands before the CTA's shared memory is released
        if (q_issued > 0) mbar_wait(&sm.q_full, (q_issued - 1) & 1, abort, false);
        for (int j = max(0, issued - kStages); j < issued; ++j)
          mbar_wait(kq ? &sm.k_full[j % kStages] : &sm.v_full[j % kStages], (j / kStages) & 1, abort, false);
      }
    }
   } else {
    // ---------------- MMA issuers: warp 1 for query tile A, warp 2 for tile B ----------------
    // Each issues its tile's chain PV(j), QK(j + 1) from one thread (in order, so QK(j + 1)
    // overwrites S only after PV(j) read P from it); two issuing warps on different
    // sub-partitions feed the tensor pipe faster than one.  Warp 1 also zeroes the
    // invalid rows of a last V tile and then signals v_ready for warp 2.
    const int t = warp - 1;
    constexpr uint32_t kIdQK = idesc_f16(kBf16 ? 1u : 0u, 0);
    constexpr uint32_t kIdPV = idesc_f16(kBf16 ? 1u : 0u, 1);
    const uint32_t s_col = t ? 128u : 0u, o_col = t ? 384u : 256u;
    // A short last tile without the causal mask (`rem` slots in range, the same for every
    // row) is computed only as far as the softmax reads it: QK over 32 * ceil(rem / 32)
    // slots (MMA N), PV over 16 * ceil(rem / 16) slots (K steps).  The softmax stores P
    // for those columns only.
    auto trimmed = [&](int rem) { return !p.causal && rem < kBN; };
    auto issue_qk = [&](int s, int rem) {
      const SDesc qd = sdesc2(smem_u32(sm.q[t]), 16, 1024), kd = sdesc2(smem_u32(sm.k[s]), 16, 1024);
      const uint32_t idesc =
          trimmed(rem) ? (kIdQK & ~(0x3Fu << 17)) | ((uint32_t)(((rem + 31) / 32) * 32 >> 3) << 17) : kIdQK;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
        mma_ss2(tmem + s_col, qd, off, kd, off, idesc, kk > 0);
      }
    };
    auto pv_steps = [&](int rem) { return trimmed(rem) ? (rem + 15) / 16 : kBN / 16; };
    auto issue_pv = [&](int s, int j, int steps) {
      const SDesc vd = sdesc2(smem_u32(sm.v[s]), kBoxBytes, 1024);
      if (steps == kBN / 16) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts2(tmem + o_col, tmem + s_col + kk * 8, vd, kk * 16 * 128, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
      } else {
#pragma unroll 1
        for (int kk = 0; kk < steps; ++kk)
          mma_ts2(tmem + o_col, tmem + s_col + kk * 8, vd, kk * 16 * 128, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
      }
    };
    int T = 0, n_items_done = 0;
    RowCache rc;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      Item I;
      if (!item_geom(item, pairs, p, meta, rc, &I)) continue;
      const int s0 = T % kStages, u0 = T / kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full, n_items_done & 1, abort) &&
                                       mbar_wait(&sm.k_full[s0], u0 & 1, abort));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        issue_qk(s0, I.kv_end);
        mma_commit(&sm.s_full[t]);
        mma_commit(&sm.k_empty[s0]);
        if (I.n_tiles == 1) mma_commit(&sm.q_free);
      }
      __syncwarp();
      for (int j = 0; ok && j < I.n_tiles; ++j) {
        const int Tj = T + j, s = Tj % kStages, u = Tj / kStages;
        if (t == 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[s], u & 1, abort));
          if (!ok) break;
          const int rem = I.kv_end - j * kBN;
          if (rem < kBN) {
            // slots past the valid range may hold anything (NaN included): zero the V rows
            // the PV reads there, so that P = 0 contributes exactly nothing
            const int rows_read = pv_steps(rem) * 16;
            for (int e = lane; e < (rows_read - rem) * 2 * 8; e += 32) {
              const int r = rem + e / 16, half = (e / 8) & 1, c = e & 7;
              *reinterpret_cast<uint4*>(sm.v[s] + half * kBoxBytes + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.v_ready[s]);
        } else {
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_ready[s], u & 1, abort));
          if (!ok) break;
        }
        const bool more = j + 1 < I.n_tiles;
        const int s1 = (Tj + 1) % kStages, u1 = (Tj + 1) / kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_ready[t], Tj & 1, abort));
        if (!ok) break;
        // keep the single-issuer order PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1) at half-group
        // granularity: B's PV(j) after A issued PV(j), A's PV(j) after B issued PV(j - 1),
        // so that the two tiles stay half a period apart and their softmaxes alternate
        if (t == 1) ok = __all_sync(0xffffffffu, mbar_wait(&sm.tok[0], Tj & 1, abort));
        else if (Tj > 0) ok = __all_sync(0xffffffffu, mbar_wait(&sm.tok[1], (Tj - 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          issue_pv(s, j, pv_steps(I.kv_end - j * kBN));
          mma_commit(&sm.v_empty[s]);
          mbar_arrive(&sm.tok[t]);
        }
        if (more) {
          ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[s1], u1 & 1, abort));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
            issue_qk(s1, I.kv_end - (j + 1) * kBN);
            mma_commit(&sm.s_full[t]);
            mma_commit(&sm.k_empty[s1]);
            if (j + 2 == I.n_tiles) mma_commit(&sm.q_free);   // that was this item's last QK
          }
        } else if (lane == 0) {
          mma_commit(&sm.o_done[t]);
        }
        __syncwarp();
      }
      T += I.n_tiles;
      ++n_items_done;
    }
    if (abort->abort && lane == 0) {
      // drain: all MMAs issued by this thread complete before TMEM is released
      mma_commit(&sm.drain[t]);
      mbar_wait(&sm.drain[t], 0, abort, false);
    }
    __syncwarp();
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ---------------- softmax (one query row per thread) ----------------
    // The epilogue of an item (O / l to global memory) runs at the start of the next
    // item, while that item's Q tiles are still loading: the warp reads the previous O
    // out of TMEM (once its last PV is done), stores it, and only then waits for the new
    // item's first S tile.  Its first P-ready, which follows in program order, also tells
    // the issuer that O is free for the new item's first PV.
    const int t = (warp - 4) >> 2;          // query tile A or B
    const int quad = warp & 3;              // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;         // row within the tile
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t s_addr = lane_addr + (t ? 128u : 0u);
    const uint32_t o_addr = lane_addr + (t ? 384u : 256u);
    const float c = p.scale_log2;
    uint8_t* const stage = sm.o_stage[warp - 4][0];
    int T = 0, n_items_done = 0;
    RowCache rc;
    bool ok = true;
    // the item whose output is still in O: its head, batch row, first row of this warp, this
    // thread's query row, and the row's running max and sum
    bool pend = false;
    int pend_b = 0, pend_h = 0, pend_grow = 0, pend_row = 0;
    float pend_m = 0.f, pend_l = 0.f;
    // The pending item's output: once its last PV is done, O / l leaves TMEM 64 columns at
    // a time through the warp's two 64-byte-swizzled staging buffers (16-byte chunk c of
    // row r at chunk c ^ ((r >> 1) & 3), conflict-free), one proxy fence and two 32-column
    // TMA stores per 64 columns; rows past n_q are clipped by the map.  Also the LSE of
    // the row.
    auto o_flush = [&]() {
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&sm.o_done[t], (n_items_done - 1) & 1, abort));
      if (!ok) return;
      tc_fence_after();
      const float inv = pend_l > 0.f ? 1.f / pend_l : 0.f;
      if (p.lse != nullptr && pend_row < p.n_q)   // m and l are in the exp2 domain of scale * q.k
        p.lse[((int64_t)pend_b * p.n_q + pend_row) * g.H + pend_h] =
            pend_l > 0.f ? (pend_m + log2f(pend_l)) * 0.6931471805599453f : -INFINITY;
      // two halves of 64 columns: both staging buffers filled, one proxy fence, two stores
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t orow[64];
        tmem_ld32(o_addr + hf * 64, orow);
        tmem_ld32(o_addr + hf * 64 + 32, orow + 32);
        tmem_ld_wait();
        reg_fence32(orow);
        reg_fence32(orow + 32);
        if (lane == 0) bulk_wait_read0();              // the stores that last read both buffers are done
        __syncwarp();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 y = __fmul2_rn(
                make_float2(__uint_as_float(orow[c2 * 32 + 2 * i]), __uint_as_float(orow[c2 * 32 + 2 * i + 1])),
                make_float2(inv, inv));
            pk[i] = pack2<kBf16>(y.x, y.y);
          }
          uint8_t* buf = stage + c2 * kStageBytes;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) * 16)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          const int c1 = 2 * hf + 1;                   // the half's second 32-column box
          tma_store_4d(&tm_o, stage, hf * 64, pend_h, pend_grow, pend_b);
          tma_store_4d(&tm_o, stage + kStageBytes, c1 * 32, pend_h, pend_grow, pend_b);
          bulk_commit();
        }
      }
    };
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      Item I;
      if (!item_geom(item, pairs, p, meta, rc, &I)) continue;
      const int row = I.row_a + t * kBM + r;   // query row within the chunk
      const int qpos = I.qpos0 + row;
      float m_ref = -INFINITY, l = 0.f;
      if (pend) {
        o_flush();
        if (!ok) break;
        pend = false;
      }
      for (int j = 0; j < I.n_tiles; ++j) {
        const int Tj = T + j;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], Tj & 1, abort));
        if (!ok) break;
        tc_fence_after();
        int valid = I.kv_end - j * kBN;                          // columns < valid are slots in range
        if (p.causal) valid = min(valid, qpos - j * kBN + 1);
        // One pass over the tile's S row: kChunks 32-column chunks hold slots in range
        // (fewer than 4 only on a short last tile without the causal mask, where
        // `valid` is the same for every row and the MMAs cover only those chunks);
        // kMask masks columns past `valid`.
        auto tile = [&](auto chunks, auto mask) {
          constexpr int kC = decltype(chunks)::value;
          constexpr bool kM = decltype(mask)::value;
          uint32_t sr[128];
#pragma unroll
          for (int q4 = 0; q4 < kC; ++q4) tmem_ld32(s_addr + q4 * 32, sr + q4 * 32);
          tmem_ld_wait();
#pragma unroll
          for (int q4 = 0; q4 < kC; ++q4) reg_fence32(sr + q4 * 32);
          const float m_tile = row_max<kM, kC>(sr, valid) * c;
          bool rescale = m_tile > m_ref + kRescaleThreshold;
          const float m_new = rescale ? m_tile : m_ref;
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          const float alpha = rescale && j > 0 ? ex2(m_ref - m_use) : 1.f;
          m_ref = m_new;
          // P first (the S row's registers are free after it), then O *= alpha: both land
          // before this tile's P-ready, which the PV of the tile waits for
          l = l * alpha + exp_pack_store<kBf16, kM, kC, false>(sr, valid, c, m_use, s_addr);
          if (__any_sync(0xffffffffu, rescale) && j > 0) {
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t orow[32];
              tmem_ld32(o_addr + q4 * 32, orow);
              tmem_ld_wait();
              reg_fence32(orow);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 y = __fmul2_rn(make_float2(__uint_as_float(orow[i]), __uint_as_float(orow[i + 1])),
                                            make_float2(alpha, alpha));
                orow[i] = __float_as_uint(y.x);
                orow[i + 1] = __float_as_uint(y.y);
              }
              tmem_st32(o_addr + q4 * 32, orow);
            }
          }
        };
        using C1 = std::integral_constant<int, 1>;
        using C2 = std::integral_constant<int, 2>;
        using C3 = std::integral_constant<int, 3>;
        using C4 = std::integral_constant<int, 4>;
        using Masked = std::true_type;
        // Causal: `valid` differs between rows, and the tile is unmasked only where it covers
        // every row of this warp; without the mask it is the same for all rows.
        const bool whole = p.causal ? __all_sync(0xffffffffu, valid >= kBN) : valid >= kBN;
        if (whole) {
          tile(C4{}, std::false_type{});
        } else if (p.causal || valid > 96) {
          tile(C4{}, Masked{});
        } else if (valid <= 32) {
          tile(C1{}, Masked{});
        } else if (valid <= 64) {
          tile(C2{}, Masked{});
        } else {
          tile(C3{}, Masked{});
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_ready[t]);
      }
      if (!ok) break;
      pend = true;
      pend_b = I.b;
      pend_h = I.h;
      pend_grow = I.row_a + t * kBM + quad * 32;
      pend_row = row;
      pend_m = m_ref;
      pend_l = l;
      T += I.n_tiles;
      ++n_items_done;
    }
    if (ok && pend) o_flush();
    if (lane == 0) bulk_wait_all();                      // staging stays live until the stores land
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && sm.wc.abort) atomicOr(meta + KVC_META_ERR, KVC_DEV_TIMEOUT);
}

// ---- one query tile per item: S triple-buffered in TMEM -----------------------------
// Work item = one 128-row query tile of one (batch row, q head); items run tile-fastest,
// so the CTAs working at once share a (row, head)'s K/V tiles through L2.  TMEM holds
// three S buffers and O (4 x 128 columns), and the QK and PV MMAs come from two warps on
// different sub-partitions.  S(j + 3) reuses S(j)'s columns once PV(j) has read P(j)
// from them (s_free), so the loop softmax(j) -> PV(j) -> QK(j + 3) -> softmax(j + 3)
// spans three tiles.  O is read by the epilogue before the next item's first PV
// (o_free): one bubble per item, which is small on the long rows this kernel is for.
// Warps (256 threads): 0 TMA producer of Q (one buffer, reloaded once the item's last
// QK is done) and K (three-stage ring), 3 TMA producer of V (two-stage ring), 1 QK
// issuer and TMEM owner, 2 PV issuer (and V-tail zeroing), 4-7 softmax and epilogue of
// the tile's 128 rows (warp & 3 = TMEM lane quadrant).
constexpr int kSBufs = 3;
constexpr int kKStages1 = 3, kVStages1 = 2;   // K and V ring depths
constexpr int kThreads1 = 256;

struct Smem1 {
  uint8_t q[kTileBytes];                // Q tile of the item
  uint8_t k[kKStages1][kTileBytes];
  uint8_t v[kVStages1][kTileBytes];
  uint8_t o_stage[4][2][kStageBytes];   // output staging per softmax warp (64-byte swizzle)
  uint64_t q_full, q_free;
  uint64_t k_full[kKStages1], k_empty[kKStages1];
  uint64_t v_full[kVStages1], v_empty[kVStages1];
  uint64_t s_full[kSBufs], p_ready[kSBufs], s_free[kSBufs];   // per S buffer
  uint64_t o_done, o_free;
  uint64_t pv_issued[2];                // [T & 1]: a phase per two tiles, PV(T)'s MMAs are being queued
  uint64_t drain[2];
  uint32_t tmem_base;
  WaitCtl wc;
};
static_assert(sizeof(Smem1) + 1024 <= 232448, "shared memory above the 227 KB a block may opt into");
static_assert(offsetof(Smem1, o_stage) % 1024 == 0, "staging buffers must keep the swizzle phase of their address");

__device__ __forceinline__ bool item_geom1(int item, int qtiles, const TcParams& p, int32_t* meta, RowCache& rc,
                                           Item* it) {
  const kvc_geom& g = p.g;
  const int qt = item % qtiles, bh = item / qtiles;
  it->h = bh % g.H;
  it->b = bh / g.H;
  it->kvh = it->h / (g.H / g.Hkv);
  it->row_a = qt * kBM;
  if (it->b != rc.b) {
    rc.b = it->b;
    rc.ok = kvc_row_range(g, it->b, &rc.row0, &rc.len, meta + KVC_META_ERR);
  }
  if (!rc.ok) return false;
  const int len = rc.len;
  it->row0 = rc.row0;
  it->kv_batch = g.layout == KVC_PACKED ? 0 : it->b;
  it->qpos0 = len - p.n_q;
  it->kv_end = len;
  if (p.causal) {
    const int last_row = min(it->row_a + kBM, p.n_q) - 1;
    it->kv_end = max(1, min(len, it->qpos0 + last_row + 1));
  }
  it->n_tiles = (it->kv_end + kBN - 1) / kBN;
  return true;
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads1, 1)
k_attn_1q(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
          int32_t* __restrict__ meta, TcParams p) {
  kvc_pdl_wait();   // launched as a programmatic dependent: nothing is read before this
  kvc_pdl_release();
  extern __shared__ uint8_t smem_raw[];
  Smem1& sm = *reinterpret_cast<Smem1*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const kvc_geom& g = p.g;
  const int qtiles = (p.n_q + kBM - 1) / kBM;
  const int n_items = g.B * g.H * qtiles;

  if (threadIdx.x == 0) {
    sm.wc.abort = (*reinterpret_cast<volatile int32_t*>(meta + KVC_META_ERR) & KVC_DEV_TIMEOUT) ? 1 : 0;
    sm.wc.limit_ns = p.stall_ns > 0 ? p.stall_ns : kTimeoutNs;
    sm.wc.stall = p.stall_ns > 0;
  }
  __syncthreads();
  if (sm.wc.abort) return;
  volatile WaitCtl* abort = &sm.wc;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_free, 1);
    for (int b = 0; b < 2; ++b) mbar_init(&sm.drain[b], 1);
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_ready[b], kBM / 32);   // one arrival per softmax warp
      mbar_init(&sm.s_free[b], 1);
    }
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.o_free, kBM / 32);
    for (int b = 0; b < 2; ++b) mbar_init(&sm.pv_issued[b], 1);
    for (int s = 0; s < kKStages1; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages1; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    mbar_init(&sm.wc.never, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0 || warp == 3) {
    // ---------------- TMA producers: warp 0 Q and K, warp 3 V ----------------
    // (two threads, so that a K load never queues behind a V load waiting for a PV)
    if (lane == 0) {
      const bool kq = warp == 0;
      const int stages = kq ? kKStages1 : kVStages1;
      int T = 0, n = 0;
      RowCache rc;
      int issued = 0, q_issued = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        Item I;
        if (!item_geom1(item, qtiles, p, meta, rc, &I)) continue;
        if (kq) {
          if (n >= 1 && !mbar_wait(&sm.q_free, (n - 1) & 1, abort)) break;   // item n - 1's last QK
          mbar_expect_tx(&sm.q_full, kTileBytes);
          for (int half = 0; half < 2; ++half)
            tma_load_4d(&tm_q, &sm.q_full, sm.q + half * kBoxBytes, half * 64, I.h, I.row_a, I.b);
          q_issued = n + 1;
        }
        const CUtensorMap* tm = kq ? &tm_k : &tm_v;
        for (int j = 0; j < I.n_tiles; ++j) {
          const int Tj = T + j, s = Tj % stages, u = Tj / stages;
          uint64_t* empty = kq ? &sm.k_empty[s] : &sm.v_empty[s];
          uint64_t* full = kq ? &sm.k_full[s] : &sm.v_full[s];
          uint8_t* dst = kq ? sm.k[s] : sm.v[s];
          if (Tj >= stages && !mbar_wait(empty, (u - 1) & 1, abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full, kTileBytes);
          for (int half = 0; half < 2; ++half)
            tma_load_4d(tm, full, dst + half * kBoxBytes, half * 64, I.kvh, I.row0 + j * kBN, I.kv_batch);
          issued = Tj + 1;
        }
        T += I.n_tiles;
        ++n;
      }
      if (abort->abort) {
        // drain: every load this thread issued lands before the CTA's shared memory is released
        if (q_issued > 0) mbar_wait(&sm.q_full, (q_issued - 1) & 1, abort, false);
        for (int j = max(0, issued - stages); j < issued; ++j)
          mbar_wait(kq ? &sm.k_full[j % stages] : &sm.v_full[j % stages], (j / stages) & 1, abort, false);
      }
    }
  } else if (warp == 1) {
    // ---------------- QK issuer: S(T) = Q K(T)^T into S buffer T % 2 ----------------
    constexpr uint32_t kIdQK = idesc_f16(kBf16 ? 1u : 0u, 0);
    int T = 0, n = 0;
    RowCache rc;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      Item I;
      if (!item_geom1(item, qtiles, p, meta, rc, &I)) continue;
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full, n & 1, abort));
      for (int j = 0; ok && j < I.n_tiles; ++j) {
        const int Tj = T + j, s = Tj % kKStages1, u = Tj / kKStages1, sb = Tj % kSBufs;
        // K(T) landed, S buffer sb is free (PV(T - 3) read its P), and PV(T - 2) is being
        // issued (the PV issuer signals once half its MMAs are queued, so that this
        // thread's wake-up overlaps the rest and the tensor pipe does not drain between
        // the two): the queue then alternates PV(T - 2), QK(T), PV(T - 1), ... rather
        // than holding QKs issued far ahead in front of the PV a softmax is waiting on.
        // (PV(T - 1) may be signalled too by then, so the token alternates between two
        // barriers: a phase parity on one barrier could not tell T - 2 from T.)
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[s], u & 1, abort) &&
                                         (Tj < kSBufs || mbar_wait(&sm.s_free[sb], (Tj / kSBufs - 1) & 1, abort)) &&
                                         (Tj < 2 || mbar_wait(&sm.pv_issued[Tj & 1], ((Tj - 2) >> 1) & 1, abort)));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const SDesc qd = sdesc2(smem_u32(sm.q), 16, 1024), kd = sdesc2(smem_u32(sm.k[s]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            mma_ss2(tmem + sb * 128u, qd, off, kd, off, kIdQK, kk > 0);
          }
          mma_commit(&sm.s_full[sb]);
          mma_commit(&sm.k_empty[s]);
          if (j + 1 == I.n_tiles) mma_commit(&sm.q_free);
        }
        __syncwarp();
      }
      T += I.n_tiles;
      ++n;
    }
    if (abort->abort && lane == 0) {
      mma_commit(&sm.drain[0]);
      mbar_wait(&sm.drain[0], 0, abort, false);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---------------- PV issuer: O(item) += P(T) V(T) ----------------
    constexpr uint32_t kIdPV = idesc_f16(kBf16 ? 1u : 0u, 1);
    int T = 0, n = 0;
    RowCache rc;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      Item I;
      if (!item_geom1(item, qtiles, p, meta, rc, &I)) continue;
      // O is free once the epilogue of item n - 1 has read it
      ok = __all_sync(0xffffffffu, n < 1 || mbar_wait(&sm.o_free, (n - 1) & 1, abort));
      for (int j = 0; ok && j < I.n_tiles; ++j) {
        const int Tj = T + j, s = Tj % kVStages1, u = Tj / kVStages1, sb = Tj % kSBufs;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[s], u & 1, abort));
        if (!ok) break;
        const int rem = I.kv_end - j * kBN;
        if (rem < kBN) {
          // slots past the valid range may hold anything (NaN included): zero those V rows
          // so that P = 0 there contributes exactly nothing
          for (int e = lane; e < (kBN - rem) * 2 * 8; e += 32) {
            const int r = rem + e / 16, half = (e / 8) & 1, c = e & 7;
            *reinterpret_cast<uint4*>(sm.v[s] + half * kBoxBytes + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
          __syncwarp();
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_ready[sb], (Tj / kSBufs) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const SDesc vd = sdesc2(smem_u32(sm.v[s]), kBoxBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            mma_ts2(tmem + 384u, tmem + sb * 128u + kk * 8, vd, kk * 16 * 128, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
            if (kk == 3) mbar_arrive(&sm.pv_issued[Tj & 1]);
          }
          mma_commit(&sm.s_free[sb]);
          mma_commit(&sm.v_empty[s]);
          if (j + 1 == I.n_tiles) mma_commit(&sm.o_done);
        }
        __syncwarp();
      }
      T += I.n_tiles;
      ++n;
    }
    if (abort->abort && lane == 0) {
      mma_commit(&sm.drain[1]);
      mbar_wait(&sm.drain[1], 0, abort, false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- softmax and epilogue (one query row per thread) ----------------
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const float c = p.scale_log2;
    uint8_t* const stage = sm.o_stage[quad][0];
    int T = 0, n = 0;
    RowCache rc;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      Item I;
      if (!item_geom1(item, qtiles, p, meta, rc, &I)) continue;
      const uint32_t o_addr = lane_addr + 384u;
      const int row = I.row_a + r;
      const int qpos = I.qpos0 + row;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < I.n_tiles; ++j) {
        const int Tj = T + j, sb = Tj % kSBufs;
        const uint32_t s_addr = lane_addr + sb * 128u;
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[sb], (Tj / kSBufs) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        int valid = I.kv_end - j * kBN;
        if (p.causal) valid = min(valid, qpos - j * kBN + 1);
        auto tile = [&](auto chunks, auto mask) {
          constexpr int kC = decltype(chunks)::value;
          constexpr bool kM = decltype(mask)::value;
          uint32_t sr[128];
#pragma unroll
          for (int q4 = 0; q4 < kC; ++q4) tmem_ld32(s_addr + q4 * 32, sr + q4 * 32);
          tmem_ld_wait();
#pragma unroll
          for (int q4 = 0; q4 < kC; ++q4) reg_fence32(sr + q4 * 32);
          // After the first tile, P is computed at once against the current reference
          // max.  Every p of the row is at most the row's sum of p, so a sum of at most
          // 2^threshold shows that the tile's max did not grow by more than the threshold
          // and P stands (the common case, which needs no max pass).  Otherwise (rare)
          // the tile's max is found and the tile redone against it where it grew by more
          // than the threshold: the same rescale decisions, and so the same result, as
          // testing the tile's max itself.
          float lsum = 0.f;
          if (j > 0) {
            lsum = exp_pack_store<kBf16, kM, kC>(sr, valid, c, m_ref, s_addr);
            if (!__any_sync(0xffffffffu, !(lsum <= kRescaleSum))) {   // (a NaN sum takes the slow path)
              l += lsum;
              return;
            }
          }
          const float m_tile = row_max<kM, kC>(sr, valid) * c;
          const bool rescale = m_tile > m_ref + kRescaleThreshold;
          const float m_new = rescale ? m_tile : m_ref;
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          if (j > 0) {
            tmem_st_wait();                                // the optimistic P is overwritten below
            // O may be rescaled only once PV(T - 1) has finished accumulating into it
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_free[(Tj - 1) % kSBufs], ((Tj - 1) / kSBufs) & 1, abort)))
              return;
            tc_fence_after();
            const float alpha = rescale ? ex2(m_ref - m_use) : 1.f;
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t orow[32];
              tmem_ld32(o_addr + q4 * 32, orow);
              tmem_ld_wait();
              reg_fence32(orow);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 y = __fmul2_rn(make_float2(__uint_as_float(orow[i]), __uint_as_float(orow[i + 1])),
                                            make_float2(alpha, alpha));
                orow[i] = __float_as_uint(y.x);
                orow[i + 1] = __float_as_uint(y.y);
              }
              tmem_st32(o_addr + q4 * 32, orow);
            }
            tmem_st_wait();
            l *= alpha;
          }
          m_ref = m_new;
          l += exp_pack_store<kBf16, kM, kC>(sr, valid, c, m_use, s_addr);
        };
        using C1 = std::integral_constant<int, 1>;
        using C2 = std::integral_constant<int, 2>;
        using C3 = std::integral_constant<int, 3>;
        using C4 = std::integral_constant<int, 4>;
        using Masked = std::true_type;
        // Causal: `valid` differs between rows, and the tile is unmasked only where it covers
        // every row of this warp; without the mask it is the same for all rows.
        const bool whole = p.causal ? __all_sync(0xffffffffu, valid >= kBN) : valid >= kBN;
        if (whole) {
          tile(C4{}, std::false_type{});
        } else if (p.causal || valid > 96) {
          tile(C4{}, Masked{});
        } else if (valid <= 32) {
          tile(C1{}, Masked{});
        } else if (valid <= 64) {
          tile(C2{}, Masked{});
        } else {
          tile(C3{}, Masked{});
        }
        if (abort->abort) {
          ok = false;
          break;
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_ready[sb]);
      }
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&sm.o_done, n & 1, abort));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (p.lse != nullptr && row < p.n_q)   // m_ref and l are in the exp2 domain of scale * q.k
        p.lse[((int64_t)I.b * p.n_q + row) * g.H + I.h] =
            l > 0.f ? (m_ref + log2f(l)) * 0.6931471805599453f : -INFINITY;
      const int grow = I.row_a + quad * 32;    // first query row of this warp
#pragma unroll 1
      for (int q2 = 0; q2 < 2; ++q2) {                  // 64 columns per TMEM round trip
        uint32_t orow[64];
        tmem_ld32(o_addr + q2 * 64, orow);
        tmem_ld32(o_addr + q2 * 64 + 32, orow + 32);
        tmem_ld_wait();
        reg_fence32(orow);
        reg_fence32(orow + 32);
        if (lane == 0) bulk_wait_read0();              // the stores that last read both buffers are done
        __syncwarp();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {               // both staging buffers, then one proxy fence
          const uint32_t* oc = orow + 32 * c2;
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 y = __fmul2_rn(make_float2(__uint_as_float(oc[2 * i]), __uint_as_float(oc[2 * i + 1])),
                                        make_float2(inv, inv));
            pk[i] = pack2<kBf16>(y.x, y.y);
          }
          uint8_t* buf = stage + c2 * kStageBytes;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) * 16)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          const int c1 = 2 * q2 + 1;                   // the half's second 32-column box
          tma_store_4d(&tm_o, stage, q2 * 64, I.h, grow, I.b);
          tma_store_4d(&tm_o, stage + kStageBytes, c1 * 32, I.h, grow, I.b);
          bulk_commit();
        }
      }
      // every TMEM read of O is complete: item n + 1's first PV may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.o_free);
      T += I.n_tiles;
      ++n;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && sm.wc.abort) atomicOr(meta + KVC_META_ERR, KVC_DEV_TIMEOUT);
}

// ---- host side ----------------------------------------------------------------
bool make_map(CUtensorMap* m, int dtype, const void* base, uint64_t d1, uint64_t d2, uint64_t d3) {
  return kvc_make_tile_map(m, dtype, base, kD, d1, d2, d3, 128);
}

size_t smem_bytes() { return sizeof(Smem) + 1024; }
size_t smem_bytes1() { return sizeof(Smem1) + 1024; }

}  // namespace

bool kvc_tc_supported(const kvc_config& cfg) {
  return (cfg.dtype == KVC_BF16 || cfg.dtype == KVC_F16) && cfg.head_dim == kD;
}

bool kvc_tc_make_kv_maps(kvc_cache* c) {
  const kvc_config& g = c->cfg;
  const uint64_t rows = (uint64_t)c->cap;
  const uint64_t batches = g.layout == KVC_PACKED ? 1 : (uint64_t)g.batch;
  if (!make_map(&c->tm_k, g.dtype, c->k, g.kv_heads, rows, batches)) return false;
  if (!make_map(&c->tm_v, g.dtype, c->v, g.kv_heads, rows, batches)) return false;
  const size_t smem = smem_bytes();
  if (cudaFuncSetAttribute(k_attn_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(k_attn_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return false;
  const size_t smem1 = smem_bytes1();
  if (cudaFuncSetAttribute(k_attn_1q<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(k_attn_1q<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess)
    return false;
  return true;
}

namespace {
// The pair kernel's register split needs every thread launched with kRegsLaunch registers.
bool pair_regs_ok() {
  static int ok = -1;
  if (ok < 0) {
    cudaFuncAttributes a{}, b{};
    ok = cudaFuncGetAttributes(&a, k_attn_tc<true>) == cudaSuccess &&
         cudaFuncGetAttributes(&b, k_attn_tc<false>) == cudaSuccess && a.numRegs == (int)kRegsLaunch &&
         b.numRegs == (int)kRegsLaunch;
  }
  return ok == 1;
}
}  // namespace

cudaError_t kvc_launch_attn_tc(kvc_cache* c, const void* q, void* out, int n_q, bool causal, float* lse,
                               cudaStream_t s) {
  const kvc_config& cfg = c->cfg;
  CUtensorMap tm_q;
  CUtensorMap tm_o;
  if (!make_map(&tm_q, cfg.dtype, q, cfg.heads, (uint64_t)n_q, cfg.batch)) return cudaErrorInvalidValue;
  if (!kvc_make_tile_map(&tm_o, cfg.dtype, out, kD, cfg.heads, (uint64_t)n_q, cfg.batch, 32, KVC_BOX_SW64))
    return cudaErrorInvalidValue;
  TcParams p;
  p.g = kvc_geom{cfg.batch, cfg.heads, cfg.kv_heads, cfg.head_dim, c->cap, cfg.layout, c->lens};
  p.n_q = n_q;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = c->scale * 1.4426950408889634f;
  p.lse = lse;
  p.stall_ns = c->debug_stall_ns;
  // Kernel by shape (a captured graph stays valid at any length): stores whose rows hold
  // at most kShortKv slots (the whole store for PACKED) give items of a few K/V tiles,
  // where the pair kernel's eight softmax warps keep the per-item chain short; longer
  // stores run the one-tile kernel, whose triple-buffered S keeps the tensor pipe fed
  // (measured crossover between 512 and 1024 slots).
  if (c->cap <= kShortKv) {
    if (!pair_regs_ok()) return cudaErrorInvalidConfiguration;
    const int64_t items = (int64_t)((n_q + 2 * kBM - 1) / (2 * kBM)) * cfg.heads * cfg.batch;
    if (items > INT32_MAX) return cudaErrorInvalidValue;
    dim3 grid((unsigned)(items < c->num_sms ? items : c->num_sms));
    if (cfg.dtype == KVC_BF16)
      return kvc_launch_pdl(k_attn_tc<true>, grid, dim3(kThreads), smem_bytes(), s, tm_q, c->tm_k, c->tm_v, tm_o,
                            c->meta, p);
    return kvc_launch_pdl(k_attn_tc<false>, grid, dim3(kThreads), smem_bytes(), s, tm_q, c->tm_k, c->tm_v, tm_o,
                          c->meta, p);
  }
  const int64_t items = (int64_t)((n_q + kBM - 1) / kBM) * cfg.heads * cfg.batch;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(items < c->num_sms ? items : c->num_sms));    // persistent: one CTA per SM
  if (cfg.dtype == KVC_BF16)
    return kvc_launch_pdl(k_attn_1q<true>, grid, dim3(kThreads1), smem_bytes1(), s, tm_q, c->tm_k, c->tm_v, tm_o,
                          c->meta, p);
  return kvc_launch_pdl(k_attn_1q<false>, grid, dim3(kThreads1), smem_bytes1(), s, tm_q, c->tm_k, c->tm_v, tm_o,
                        c->meta, p);
}
