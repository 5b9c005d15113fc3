/*
 * kvc.h — attention of a query chunk or a decode token over a device-resident
 * KV cache, on one NVIDIA GB300 (sm_103a).  C ABI of libkvc.so.
 *
 * Sources of the operations (web pages; cited by title and section):
 *  [IDX]  lingbot-world PR "refactor(kv): index_copy_ for KV-cache writes" —
 *         Summary; "What this is and isn't" (homogeneous multi-user batching,
 *         CUDA Graphs).
 *  [RING] flashdreams issue "add an opt-in circular KV policy for streaming
 *         attention" — "current path", "proposed boundary", "first experiment".
 *  [PFX]  fish-speech PR "perf(text2semantic): pass only active KV cache prefix
 *         to SDPA" — "Problem", "Change", the regression-test reply.
 *  [VAR]  TensorRT-LLM PR "FA4 variable-length cross-attention" — Description,
 *         "Microbenchmark, cross-attention op only".
 *
 * Conventions shared by every entry point
 *  - All pointers named d_* or documented "device" are device pointers; every
 *    tensor pointer must be 16-byte aligned.  Tensors are dense row-major:
 *      queries / outputs   q, out   [B, n, H, D]
 *      written K / V rows  k, v     [B, n, Hkv, D]
 *      LINEAR / CIRCULAR store      [B, cap, Hkv, D]   (cap = capacity or window)
 *      PACKED store                 [total, Hkv, D]    (row b at cu_seqlens[b])
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *    only enqueues work on it; none reads device data back on the host, so the
 *    advance / write / attend sequence can be captured in a CUDA graph once and
 *    replayed [RING "proposed boundary", IDX item 2].  kvc_get_error is the one
 *    call that synchronises.
 *  - Ownership: the caller owns and allocates every device buffer (K/V store,
 *    meta block, workspace, inputs, outputs).  The library allocates no device
 *    memory; it owns only the host-side handle.  Buffers must outlive the handle.
 *  - Counts (n_q, n_tokens, n_rows, rope_positions) must be at least 1: an empty
 *    call is KVC_ERR_ARG, not a no-op, so that a caller's off-by-one surfaces.
 *  - Return value: 0 on success, a negative KVC_ERR_* code otherwise.  Host-side
 *    validation failures enqueue nothing.  Errors found on the device (a slot,
 *    length or offset out of range) never fault: the kernel skips the offending
 *    row, sets a bit in the meta block's error word, and kvc_get_error reports it.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  F32 attention runs in true fp32 FMA arithmetic; F16/BF16 run the
 * contractions on the tensor cores with fp32 accumulation.  Outputs have the
 * input type. */
typedef enum { KVC_F32 = 0, KVC_F16 = 1, KVC_BF16 = 2 } kvc_dtype;

/* Store layouts.
 *  LINEAR   capacity slots per row, active prefix kv_len [PFX "Change"].
 *  CIRCULAR sink + rolling window of whole chunks, attended in physical order
 *           [RING "proposed boundary"]; `window` counts the sink.
 *  PACKED   ragged per-row K/V back to back, offsets cu_seqlens [VAR Description]. */
typedef enum { KVC_LINEAR = 0, KVC_CIRCULAR = 1, KVC_PACKED = 2 } kvc_layout;

typedef struct kvc_config {
  int32_t batch;       /* B rows (users / CFG branches), each with its own state   */
  int32_t heads;       /* H query heads                                            */
  int32_t kv_heads;    /* Hkv; H % Hkv == 0, q-head h reads kv-head h / (H/Hkv)     */
  int32_t head_dim;    /* D: 64 or 128                                             */
  int32_t sink;        /* CIRCULAR: pinned sink tokens, a multiple of chunk (may be 0) */
  int32_t window;      /* CIRCULAR: total slots incl. sink, sink + a multiple of chunk */
  int32_t chunk;       /* CIRCULAR: tokens per chunk                               */
  int32_t capacity;    /* LINEAR: slots per row; PACKED: total packed slots         */
  int32_t dtype;       /* kvc_dtype                                                */
  int32_t layout;      /* kvc_layout                                               */
  float softmax_scale; /* 0 => 1/sqrt(head_dim), the SDPA default                  */
} kvc_config;

typedef struct kvc_cache kvc_cache;

enum {
  KVC_OK = 0,
  KVC_ERR_ARG = -1,         /* null / misaligned pointer, bad shape or config       */
  KVC_ERR_UNSUPPORTED = -2, /* a valid request this library does not serve, e.g.
                               causal attention over a circular store [RING]       */
  KVC_ERR_RANGE = -3,       /* a host-known length out of range [PFX tests item 2] */
  KVC_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed                */
  KVC_ERR_DEVICE = -5       /* kvc_get_error: the device error word was non-zero   */
};

/* Bits of the device error word (meta word 0), reported by kvc_get_error. */
enum {
  KVC_DEV_BAD_SLOT = 1,     /* a d_slots entry outside [0, cap)                     */
  KVC_DEV_BAD_KVLEN = 2,    /* a kv_len outside [1, cap] at attend / set_lengths   */
  KVC_DEV_BAD_CUSEQ = 4,    /* cu_seqlens not increasing from 0 or beyond capacity  */
  KVC_DEV_OVERFLOW = 8,     /* LINEAR advance past capacity                         */
  KVC_DEV_NO_CHUNK = 16,    /* write with no reserved chunk                         */
  KVC_DEV_TIMEOUT = 32,     /* a bounded in-kernel wait gave up (the kernel returned) */
  KVC_DEV_BAD_POS = 64      /* kvc_write_rope: a token position outside the rope table  */
};

/* Attention flags. */
enum {
  KVC_CAUSAL = 1,           /* LINEAR only: query i at position kv_len - n_q + i sees
                               keys at positions <= its own [PFX "Change"]          */
  KVC_KERNEL_SIMT = 256,    /* run the fp32-FMA kernel for any dtype (a cross-check
                               of the tensor-core and decode kernels)               */
  KVC_DETERMINISTIC = 512   /* decode (n_q == 1): give every block a fixed set of tiles.
                               Without it, rows longer than 4 x the split count spread
                               their later tiles to whichever blocks stream fastest, so
                               the last bits of the result can vary between calls   */
};

/* Meta block: int32 words, device memory owned by the caller.
 *   [0] error word  [1..3] reserved
 *   [4 + 4b + 0] chunks reserved by row b   [4 + 4b + 1] first slot of its chunk
 *   [4 + 4b + 2] slots filled               [4 + 4b + 3] kv_len (active prefix)
 *   [4 + 4B + b], b = 0..B: cu_seqlens (PACKED)
 * kvc_create initialises it. */
size_t kvc_meta_bytes(const kvc_config* cfg);

/* Device scratch for the split-KV decode kernel (partial outputs and their
 * log-sum-exp terms, plus per-(row, kv-head) ticket and tile-claim counters that
 * each call leaves at zero).
 * Zero for a config with nothing to split.  Caller-allocated, passed to kvc_create. */
size_t kvc_workspace_bytes(const kvc_config* cfg);

/* Create a handle over caller-owned device buffers.
 *  k_store, v_store: the K and V stores (layouts above), any prior contents.
 *  meta: kvc_meta_bytes(cfg) bytes; workspace: kvc_workspace_bytes(cfg) bytes
 *  (NULL allowed when that is 0).  Enqueues the meta initialisation on `stream`:
 *  every row empty, no chunk reserved, error word 0.
 *  Errors: KVC_ERR_ARG for a bad config or pointer, KVC_ERR_UNSUPPORTED for an
 *  unsupported head_dim or dtype, KVC_ERR_CUDA. */
int kvc_create(const kvc_config* cfg, void* k_store, void* v_store, void* meta,
               void* workspace, void* stream, kvc_cache** out);

/* Reserve the next chunk of `row` (all rows when row < 0) [RING "proposed
 * boundary": reservation separate from writes, so denoising rewrites replace the
 * same chunk].
 *  CIRCULAR: n_tokens must equal `chunk`.  Chunk k's first slot is k*chunk while
 *    the ring fills, then sink + ((k - sink/chunk) mod ((window-sink)/chunk))*chunk:
 *    the oldest rolling chunk is evicted, the sink stays pinned [RING "current
 *    path"].  kv_len = min((k+1)*chunk, window).
 *  LINEAR: reserves n_tokens slots after those filled; kv_len = slots filled.  Past
 *    capacity sets KVC_DEV_OVERFLOW and leaves the row unchanged.
 *  PACKED: KVC_ERR_UNSUPPORTED (lengths come from kvc_set_lengths). */
int kvc_advance(kvc_cache* c, int32_t row, int32_t n_tokens, void* stream);

/* Write n_tokens rows of K and V (device, [B, n_tokens, Hkv, D]) into the store,
 * the index_copy-style write of [IDX Summary].
 *  d_slots == NULL: row b's token i goes to its reserved chunk (first slot from the
 *    meta block, so a replayed graph writes the slot the device holds [RING]); for
 *    PACKED to cu_seqlens[b] + i for i < len_b (the pack of [VAR]), tokens past
 *    len_b are ignored (so n_tokens may exceed a row's length, or the capacity).
 *  d_slots != NULL (device int32[n_tokens]): token i of every row goes to slot
 *    d_slots[i] — one index shared by all rows on the same timeline [IDX item 1].
 *    Not for PACKED.  Entries outside [0, cap) set KVC_DEV_BAD_SLOT and are skipped.
 * Bytes are copied unchanged (bit-exact).
 * Errors: KVC_ERR_RANGE when n_tokens exceeds the per-row slot count (not PACKED) or
 * 2 x B x n_tokens exceeds INT32_MAX;
 * KVC_ERR_ARG for a circular write whose n_tokens differs from `chunk`. */
int kvc_write(kvc_cache* c, const void* k, const void* v, int32_t n_tokens,
              const int32_t* d_slots, void* stream);

/* Append n_tokens rows of K and V (device, [B, n_tokens, Hkv, D]) to every row of a
 * LINEAR store: the same as kvc_advance(c, -1, n_tokens) followed by
 * kvc_write(c, k, v, n_tokens, NULL), in one launch when the K and V bytes appended are
 * at most 128 KiB (a decode step: the new token of each row goes to slot kv_len and the
 * row then attends kv_len + 1 slots [PFX "Change"]), as those two launches otherwise.  Slots come from
 * the meta block on the device, so a captured step appends at the right place on every
 * replay.  A row that would pass its capacity sets KVC_DEV_OVERFLOW and is left
 * unchanged.  Errors: KVC_ERR_UNSUPPORTED for CIRCULAR / PACKED (whose slots are
 * reserved per chunk or come from cu_seqlens), KVC_ERR_RANGE for n_tokens above the
 * capacity, KVC_ERR_ARG, KVC_ERR_CUDA. */
int kvc_append(kvc_cache* c, const void* k, const void* v, int32_t n_tokens, void* stream);

/* One decode step in one launch: append one token per row (k_new, v_new: device,
 * [B, 1, Hkv, D], 16-byte aligned) and attend q (device [B, 1, H, D]) over every row's
 * stored prefix plus that token, writing out (device [B, 1, H, D]).  The same result as
 * kvc_append(c, k_new, v_new, 1) followed by kvc_attend(c, q, out, 1, 0) — the store and
 * the meta block end identical; out agrees up to rounding, since the new token's score
 * and weight are taken in fp32 instead of through the 16-bit P of a tile — for the
 * fish-speech decode step of [PFX "Change"] (step i appends its token and attends the
 * prefix up to it).  Every block of the launch reads its row's length before the last
 * one to finish reading advances all rows (a counter in the meta block).  A row that
 * would pass its capacity sets KVC_DEV_OVERFLOW and is neither written nor attended.
 * Errors: KVC_ERR_UNSUPPORTED unless the store is LINEAR, 16-bit, served by the decode
 * kernel (head_dim 64 or 128, heads / kv_heads in {1, 2, 4, 8}) and reads its lengths
 * from its own meta block (no kvc_use_lengths layout); KVC_ERR_ARG; KVC_ERR_CUDA. */
int kvc_append_attend_decode(kvc_cache* c, const void* k_new, const void* v_new, const void* q, void* out,
                             void* stream);

/* kvc_write with RoPE fused into the K half: each K row is rotated at its absolute
 * position before it is stored; V rows are copied unchanged.  Keys stored in a circular
 * cache must carry their absolute-position rotation, applied before the write [RING
 * "proposed boundary"].
 *  d_rope (device fp32, [rope_positions][head_dim/2][2]): (cos, sin) of the angle of pair
 *    j at position p; pair j of a head is (x[2j], x[2j+1]) and turns to
 *    (x0 cos - x1 sin, x0 sin + x1 cos).  The store receives the exact value of each
 *    component for the given x and table entries, rounded once to nearest-even in the
 *    store type (for finite inputs): the same bits whichever rounding path a lane takes.
 *  Position of token i: CIRCULAR (chunks reserved - 1) * chunk + i; LINEAR the reserved
 *    base + i, or d_slots[i] when given; PACKED i (position within its row).
 * Tokens whose position is outside [0, rope_positions) are not written (K nor V) and
 * set KVC_DEV_BAD_POS.  Other rules and errors as kvc_write. */
int kvc_write_rope(kvc_cache* c, const void* k, const void* v, int32_t n_tokens, const int32_t* d_slots,
                   const float* d_rope, int32_t rope_positions, void* stream);

/* Set lengths from device arrays (either may be NULL).
 *  d_kv_len (int32[B]): LINEAR / CIRCULAR active prefix per row [PFX "Change"; the
 *    per-row used length of a padded store in VAR].  Values outside [1, cap] set
 *    KVC_DEV_BAD_KVLEN and leave that row's kv_len unchanged.
 *  d_cu_seqlens (int32[B+1]): PACKED offsets [VAR Description]; must start at 0,
 *    increase strictly and end <= capacity, else KVC_DEV_BAD_CUSEQ and nothing is
 *    changed.  Sets each row's kv_len to its length. */
int kvc_set_lengths(kvc_cache* c, const int32_t* d_kv_len, const int32_t* d_cu_seqlens,
                    void* stream);

/* Length layout shared by several handles [VAR Description: the cu_seqlens_kv of a
 * length layout are prepared once and cached, then reused by every layer and denoising
 * step; acceptance row "prepared once per length layout"].  A model with many layers
 * attending the same ragged text K/V (or the same per-row active prefixes) creates one
 * layout, sets it once per step, and points every layer's handle at it, instead of one
 * kvc_set_lengths per layer.
 *  d_block: caller-owned device memory of kvc_lengths_bytes(batch) bytes, 16-byte
 *    aligned, in the meta block's layout (error word, per-row kv_len, cu_seqlens);
 *    kvc_lengths_create enqueues its zeroing on `stream` (no row has a length yet).
 *  layout: KVC_LINEAR (per-row kv_len) or KVC_PACKED (cu_seqlens); CIRCULAR handles
 *    take their lengths from their own chunk state (KVC_ERR_UNSUPPORTED).
 *  capacity: lengths (LINEAR) or the packed total (PACKED) above it are rejected on the
 *    device as in kvc_set_lengths; every attend checks again against its own store.
 * kvc_lengths_set takes the same device arrays as kvc_set_lengths, with the same
 * checks; a bad array sets a bit in the layout's own error word, which kvc_get_error
 * of any handle using the layout reports (and clears).
 * kvc_use_lengths(c, L): from now on c's attends (and its PACKED writes) read kv_len /
 * cu_seqlens from L's block; L = NULL returns c to its own meta block.  L's batch must
 * equal c's and its capacity must not exceed c's (KVC_ERR_ARG); its layout must be c's
 * (KVC_ERR_UNSUPPORTED).  Host-side only: it enqueues nothing, and a graph captured
 * before the call keeps reading what it read when captured.  L must outlive every
 * handle using it. */
typedef struct kvc_lengths kvc_lengths;
size_t kvc_lengths_bytes(int32_t batch);
int kvc_lengths_create(int32_t batch, int32_t layout, int32_t capacity, void* d_block, void* stream,
                       kvc_lengths** out);
int kvc_lengths_set(kvc_lengths* L, const int32_t* d_kv_len, const int32_t* d_cu_seqlens, void* stream);
int kvc_use_lengths(kvc_cache* c, const kvc_lengths* L);
int kvc_lengths_destroy(kvc_lengths* L);

/* out[b, i, h, :] = sum_j softmax_j(scale * q[b,i,h,:] . k_j) v_j over row b's
 * valid slots, read in physical order with no gather or roll (unmasked attention
 * is invariant to permuting K and V rows together [RING "proposed boundary"]).
 * Valid slots: [0, kv_len_b) for LINEAR and CIRCULAR, [cu_b, cu_{b+1}) for PACKED;
 * nothing past them is read into the result [PFX "Change"].
 *  q (device [B, n_q, H, D]), out (device, same shape and dtype).
 *  flags: KVC_CAUSAL (LINEAR only, else KVC_ERR_UNSUPPORTED), KVC_KERNEL_SIMT,
 *  KVC_DETERMINISTIC.
 *  A row whose kv_len is outside [1, cap] at run time gets KVC_DEV_BAD_KVLEN and
 *  its output is left unwritten. */
int kvc_attend(kvc_cache* c, const void* q, void* out, int32_t n_q, uint32_t flags,
               void* stream);

/* kvc_attend that also writes the log-sum-exp of every query row's scaled scores:
 * d_lse[b, i, h] = ln(sum_j exp(scale * q[b,i,h,:] . k_j)) over the same slots (device
 * fp32 [B, n_q, H]; -inf for a row that sees no slot).  The forward_with_lse of [VAR];
 * with kvc_merge it composes attentions over disjoint key sets (a cache split across
 * stores, or a window not made of whole chunks).  Arguments and errors as kvc_attend. */
int kvc_attend_lse(kvc_cache* c, const void* q, void* out, float* d_lse, int32_t n_q, uint32_t flags,
                   void* stream);

/* Merge two attention results over disjoint key sets, row by row (device buffers):
 *   L = ln(e^lse_a + e^lse_b),  out = e^(lse_a - L) o_a + e^(lse_b - L) o_b.
 * o_a, o_b, out: [n_rows, head_dim] of `dtype` (kvc_dtype); lse_a, lse_b: fp32 [n_rows];
 * lse_out: fp32 [n_rows] or NULL.  out may alias o_a or o_b.  A row with both lse = -inf
 * gets out = 0 and L = -inf.  Errors: KVC_ERR_ARG, KVC_ERR_CUDA. */
int kvc_merge(int32_t dtype, int32_t n_rows, int32_t head_dim, const void* o_a, const float* lse_a,
              const void* o_b, const float* lse_b, void* out, float* lse_out, void* stream);

/* Comparator for measurement, not part of the path: the per-chunk copy that a
 * chronological sink + window store makes and the circular layout avoids [RING "current
 * path": the retained keys and values are cloned and copied back once per step].  On a
 * CIRCULAR handle's store read chronologically, K and V slots [sink + chunk, window) of
 * every row move to [sink, window - chunk) through d_scratch (clone, then copy back).
 * d_scratch: device, kvc_roll_scratch_bytes(cfg) bytes, 16-byte aligned.
 * Errors: KVC_ERR_UNSUPPORTED for other layouts, KVC_ERR_ARG, KVC_ERR_CUDA. */
size_t kvc_roll_scratch_bytes(const kvc_config* cfg);
int kvc_roll_window(kvc_cache* c, void* d_scratch, void* stream);

/* Forget the contents of `row` (all rows when row < 0): no chunk reserved, nothing
 * filled, kv_len 0; storage bytes are left as they are [RING "proposed boundary"
 * reset semantics]. */
int kvc_reset(kvc_cache* c, int32_t row, void* stream);

/* Synchronise `stream`, then return KVC_ERR_DEVICE if the device error word is
 * non-zero (its bits are stored in *bits when bits != NULL) and clear it; KVC_OK
 * otherwise.  When the word holds KVC_DEV_TIMEOUT, the decode kernel's ticket and
 * tile-claim counters in the workspace are zeroed too, so the next attend starts
 * clean. */
int kvc_get_error(kvc_cache* c, void* stream, int32_t* bits);

/* Testing hook for the failure path (not for production use).  Every wait inside the
 * tensor-core and decode attention kernels is bounded (0.5 s): when one runs out, the
 * kernel stops issuing work, lets its own copies and tensor-core operations in flight
 * finish, frees its tensor memory, sets KVC_DEV_TIMEOUT and returns, so that the context
 * stays usable.  With ns > 0, the steady-state waits of c's later attends wait instead
 * on a barrier that nothing signals, for ns nanoseconds, so that a test can make a wait
 * run out without any fault or hang; waits while draining are unchanged.  ns = 0 turns
 * the hook off.  Host-side only. */
int kvc_debug_stall_waits(kvc_cache* c, uint64_t ns);

/* Free the host handle.  Device buffers stay with the caller. */
int kvc_destroy(kvc_cache* c);

/* Static string for a return code. */
const char* kvc_strerror(int code);

/* Decode attention without any device allocation and without a handle.  The pages
 * have no counterpart: this entry point exists for callers that cannot allocate
 * device memory themselves, such as code running inside another framework's memory
 * pool, plugins whose host process owns every allocation, or a serving step that must
 * not allocate once its graphs are captured.  They cannot provide kvc_create's
 * workspace, so this call runs the split-KV decode kernel of kvc_attend (n_q == 1)
 * with its scratch in a fixed 4 MiB array inside libkvc.so, held on every GPU that
 * loads the library until the process exits.
 *  cfg: as for kvc_create (F16 / BF16, head_dim 64 or 128, H/Hkv in {1,2,4,8}).
 *  k_store, v_store, meta: the caller's store and meta block (kv_len or cu_seqlens
 *    already set, e.g. through a handle's kvc_advance / kvc_set_lengths);
 *  q: device [B, 1, H, D]; out: device [B, 1, H, D]; all 16-byte aligned.
 * Returns KVC_ERR_RANGE when the scratch would exceed 4 MiB (too many (row, kv head)
 * pairs), KVC_ERR_ARG / KVC_ERR_UNSUPPORTED as kvc_create, KVC_ERR_CUDA.  Calls no
 * cudaMalloc or cudaFree.  The first call on a device looks up the array's device
 * address (make that call before any stream capture).  Every call shares the array
 * and clears the part that must start at zero; calls that overlap on the GPU (other
 * streams, or host threads without ordering) race on it. */
int kvc_attend_decode_noalloc(const kvc_config* cfg, const void* k_store, const void* v_store,
                              int32_t* meta, const void* q, void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H_ */
