"""Plain CPU fp64 oracle for attention over a device-resident KV cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may import
this module.  It shares no code with the CUDA path: it imports NumPy only.

What it computes, and where each part comes from:

* ``ChronoCache`` keeps every cache row as a chronological history (position ->
  token row, stored in the input dtype, so it is exact).  It is the "independent
  chronological-history reference" of the flashdreams issue "add an opt-in circular KV
  policy for streaming attention" (section "first experiment").  Slot reservation
  (``advance``) is separate from writes so that repeated denoising writes replace the
  same chunk (same issue, "proposed boundary").
* ``ring_slot`` is the closed form of where a position lives in a circular
  sink+window store whose sink is pinned and whose rolling region is reused
  oldest-chunk-first (same issue, "current path" and "proposed boundary").  It is
  only used to read the GPU's physical store back in logical order.
* ``attend`` is naive softmax attention in fp64 over a materialised score row,
  ``softmax(scale * q k^T) v`` with scale = 1/sqrt(D) (the SDPA default, which the
  pages use unchanged), q-head h reading kv-head ``h // (H/Hkv)`` (the
  ``repeat_interleave`` head expansion of the fish-speech PR "pass only active KV
  cache prefix to SDPA", section "Problem").  The causal form masks key j for the
  query at absolute position p when j > p (same PR, section "Change").
* Active prefix: attention sees positions ``[0, kv_len)`` (same PR, "Change");
  packed ragged K/V: branch b sees its own ``len_b`` tokens (TensorRT-LLM PR "FA4
  variable-length cross-attention", "Description").
* ``attend_lse`` adds the log-sum-exp of each row's scaled scores and ``merge_lse``
  combines two attentions over disjoint key sets from their outputs and LSEs (the
  forward_with_lse of the same TensorRT-LLM PR); ``rope_apply`` rotates key pairs at
  their absolute positions (flashdreams issue, "proposed boundary") and ``rope_store``
  gives what a store of a given type holds after that rotation: the exact rotation
  rounded once to nearest-even (``round_to_format``); ``roll_left`` is the per-step
  copy a chronological store makes (same issue, "current path").

Parity pins (checked by ``tests/test_oracle.py``): brute-force ring simulation for
``ring_slot`` and the attended set; closed forms of attention (one key, equal keys,
a dominant key, duplicated kv heads); permutation invariance; torch's SDPA in fp64
on CPU as an independent library routine; the tiny active-prefix fixture printed in
the fish-speech PR (capacity 8, prefill 3, lengths 3,4,8, bounds 1/8 valid, 0/9
invalid); packed equal to padded-and-masked; LSE of one key and of equal keys and
torch.logsumexp; the merge of two halves equal to attention over their union; RoPE
against an independent rotation (the input generator's, from its own fp64 angles) and
its norm and relative-angle invariants; the once-rounded store values against exact
rational arithmetic (``fractions.Fraction``) on random, tie, near-tie, subnormal and
overflow cases, and against NumPy's own fp64 -> fp16 / fp32 rounding; the roll against
a deque of chunks.  The pin
tests also plant mistakes (an off-by-one slot, a wrong attended set, a wrong scale or
GQA map, a RoPE sign) and check that a pin catches each.
"""
from __future__ import annotations

import math

import numpy as np

LINEAR = "linear"
CIRCULAR = "circular"
PACKED = "packed"


# ---------------------------------------------------------------------------
# Circular sink + window storage (flashdreams issue, "proposed boundary")
# ---------------------------------------------------------------------------
def ring_slot(pos: int, sink: int, window: int) -> int:
    """Physical slot of chronological position ``pos`` in a ring of ``window`` slots.

    The first ``sink`` positions are pinned at slots ``[0, sink)``; later positions
    cycle through the rolling slots ``[sink, window)``.  ``window`` counts the sink.
    """
    if pos < sink:
        return pos
    return sink + (pos - sink) % (window - sink)


def ring_attended(end: int, sink: int, window: int) -> list[int]:
    """Chronological positions a chunk ending at ``end`` attends in a sink+window ring.

    The sink (first ``sink`` positions) plus the newest ``window - sink`` positions,
    the current chunk included.  While the ring is still filling this is ``[0, end)``.
    """
    head = list(range(0, min(sink, end)))
    tail_start = max(sink, end - (window - sink))
    return head + list(range(tail_start, end))


def roll_left(store, sink: int, window: int, chunk: int):
    """The chronological store's per-step copy: rows ``[sink + chunk, window)`` of each
    batch row move to ``[sink, window - chunk)`` (flashdreams issue, "current path");
    the rest is unchanged.  ``store``: ``[B, window, ...]``."""
    out = np.array(store, copy=True)
    out[:, sink:window - chunk] = np.asarray(store)[:, sink + chunk:window]
    return out


def check_ring_layout(sink: int, window: int, chunk: int) -> None:
    """Whole-chunk sink and window sizes, as the circular policy starts with."""
    if chunk <= 0 or window <= sink or sink < 0:
        raise ValueError("need chunk > 0, window > sink >= 0")
    if sink % chunk or (window - sink) % chunk:
        raise ValueError("sink and window - sink must be whole chunks")


# ---------------------------------------------------------------------------
# Chronological-history cache
# ---------------------------------------------------------------------------
class ChronoCache:
    """Per-row chronological history of K and V token rows.

    ``layout`` is one of LINEAR (a capacity-sized store with an active prefix
    ``kv_len``), CIRCULAR (sink + rolling window of whole chunks) or PACKED (one
    flat store holding every row's ragged K/V back to back, lengths given by
    ``cu_seqlens``).
    """

    def __init__(self, batch, kv_heads, head_dim, layout, *, sink=0, window=0,
                 chunk=0, capacity=0):
        self.batch, self.kv_heads, self.head_dim = batch, kv_heads, head_dim
        self.layout = layout
        self.sink, self.window, self.chunk, self.capacity = sink, window, chunk, capacity
        if layout == CIRCULAR:
            check_ring_layout(sink, window, chunk)
        self.reset()

    # -- lifecycle --------------------------------------------------------
    def reset(self, row: int = -1) -> None:
        rows = range(self.batch) if row < 0 else [row]
        if row < 0:
            self.hist_k = [dict() for _ in range(self.batch)]
            self.hist_v = [dict() for _ in range(self.batch)]
            self.n_chunks = [0] * self.batch
            self.chunk_start = [None] * self.batch
            self.chunk_len = [0] * self.batch
            self.filled = [0] * self.batch
            self.kv_len = [0] * self.batch
            self.cu_seqlens = None
            return
        for b in rows:
            self.hist_k[b] = {}
            self.hist_v[b] = {}
            self.n_chunks[b] = 0
            self.chunk_start[b] = None
            self.chunk_len[b] = 0
            self.filled[b] = 0
            self.kv_len[b] = 0

    def advance(self, row: int = -1, n_tokens: int | None = None) -> None:
        """Reserve the next chunk for ``row`` (all rows when ``row < 0``)."""
        rows = range(self.batch) if row < 0 else [row]
        for b in rows:
            if self.layout == CIRCULAR:
                n = self.chunk
                start = self.n_chunks[b] * self.chunk
                self.filled[b] = min(start + n, self.window)
            elif self.layout == LINEAR:
                n = int(n_tokens)
                start = self.filled[b]
                if start + n > self.capacity:
                    raise ValueError("advance past capacity")
                self.filled[b] = start + n
            else:
                raise ValueError("packed stores have no chunk reservation")
            self.chunk_start[b] = start
            self.chunk_len[b] = n
            self.n_chunks[b] += 1
            self.kv_len[b] = self.filled[b]

    def set_lengths(self, kv_len=None, cu_seqlens=None) -> None:
        if kv_len is not None:
            for b, n in enumerate(kv_len):
                n = int(n)
                cap = self.capacity if self.layout == LINEAR else self.window
                if not 1 <= n <= cap:
                    raise ValueError(f"kv_len {n} outside [1, {cap}]")
                self.kv_len[b] = n
        if cu_seqlens is not None:
            cu = [int(x) for x in cu_seqlens]
            if len(cu) != self.batch + 1 or cu[0] != 0:
                raise ValueError("cu_seqlens must have batch+1 entries starting at 0")
            for b in range(self.batch):
                if not 0 < cu[b + 1] - cu[b]:
                    raise ValueError("empty or decreasing cu_seqlens")
            if cu[-1] > self.capacity:
                raise ValueError("packed total exceeds capacity")
            self.cu_seqlens = cu
            for b in range(self.batch):
                self.kv_len[b] = cu[b + 1] - cu[b]

    def write(self, k, v, slots=None) -> None:
        """Store token rows ``k[b, i], v[b, i]`` (arrays ``[B, n, Hkv, D]``).

        Without ``slots`` row b's tokens land at the chunk it reserved (CIRCULAR,
        LINEAR) or at its first ``len_b`` positions (PACKED).  With ``slots`` (LINEAR
        only) token i of every row goes to position ``slots[i]``: one index shared by
        all rows on the same timeline (lingbot-world PR "refactor(kv): index_copy_ for
        KV-cache writes", "What this is and isn't", item 1).
        """
        k = np.asarray(k)
        v = np.asarray(v)
        n = k.shape[1]
        for b in range(self.batch):
            if slots is not None:
                if self.layout != LINEAR:
                    raise ValueError("explicit slots are positions only in a linear store")
                positions = [int(s) for s in slots]
            elif self.layout == PACKED:
                positions = list(range(min(n, self.kv_len[b])))
            else:
                if self.chunk_start[b] is None:
                    raise ValueError("write before advance")
                if n != self.chunk_len[b]:
                    raise ValueError("write size differs from the reserved chunk")
                positions = [self.chunk_start[b] + i for i in range(n)]
            for i, p in enumerate(positions):
                self.hist_k[b][p] = k[b, i].copy()
                self.hist_v[b][p] = v[b, i].copy()

    # -- views ------------------------------------------------------------
    def attended_positions(self, b: int) -> list[int]:
        if self.layout == CIRCULAR:
            end = self.chunk_start[b] + self.chunk
            return ring_attended(end, self.sink, self.window)
        return list(range(self.kv_len[b]))

    def keys_values(self, b: int, positions=None):
        """fp64 ``[n, Hkv, D]`` K and V of row b at ``positions`` (chronological)."""
        if positions is None:
            positions = self.attended_positions(b)
        ks = np.stack([self.hist_k[b][p] for p in positions]).astype(np.float64)
        vs = np.stack([self.hist_v[b][p] for p in positions]).astype(np.float64)
        return ks, vs

    def physical_slot(self, b: int, pos: int) -> int:
        """Where the GPU store keeps position ``pos`` of row ``b``."""
        if self.layout == CIRCULAR:
            return ring_slot(pos, self.sink, self.window)
        if self.layout == PACKED:
            return self.cu_seqlens[b] + pos
        return pos


# ---------------------------------------------------------------------------
# RoPE at absolute positions (flashdreams issue, "proposed boundary": absolute positions
# determine RoPE before storage)
# ---------------------------------------------------------------------------
def rope_apply(x, positions, table):
    """Rotate pair j = (x[..., 2j], x[..., 2j+1]) of each token by the (cos, sin) that
    ``table[pos, j]`` holds, in fp64.  x: ``[n, Hkv, D]``; positions: ``[n]``.  Keys are
    rotated at their absolute position before they are stored (flashdreams issue,
    "proposed boundary")."""
    x = np.asarray(x, dtype=np.float64)
    t = np.asarray(table, dtype=np.float64)[np.asarray(positions)]      # [n, D/2, 2]
    c = t[:, None, :, 0]
    s = t[:, None, :, 1]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# Binary formats a store can hold: significand bits p (with the hidden bit), smallest
# and largest normal exponents.
FORMATS = {"bf16": (8, -126, 127), "f16": (11, -14, 15), "f32": (24, -126, 127)}


def two_sum(a, b):
    """Knuth's error-free sum in fp64: s = fl(a + b) and the exact rest e, a + b = s + e."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    s = a + b
    bb = s - a
    e = (a - (s - bb)) + (b - bb)
    return s, e


def round_to_format(hi, lo, fmt):
    """Round the exact value hi + lo (|lo| at most half an fp64 ulp of hi) to the nearest
    value of ``fmt``, ties to even, once.  Returns fp64 arrays holding those values (inf
    past the largest finite value; a zero keeps hi's sign)."""
    p, emin, emax = FORMATS[fmt]
    hi = np.asarray(hi, dtype=np.float64)
    lo = np.asarray(lo, dtype=np.float64)
    sign = np.where(np.signbit(hi), -1.0, 1.0)
    a = np.abs(hi)
    rest = lo * sign                                   # D * sign = a + rest
    _, e = np.frexp(np.where(a > 0, a, 1.0))           # a = m 2^e, m in [0.5, 1)
    q = np.maximum(e - 1, emin) - (p - 1)              # exponent of the format's spacing here
    k = np.ldexp(a, -q)                                # a in units of that spacing (exact)
    n = np.floor(k)
    frac_minus_half = (k - n) - 0.5                    # exact
    d = frac_minus_half + np.ldexp(rest, -q)           # its sign is that of the exact value's
    up = (d > 0) | ((d == 0) & (np.mod(n, 2) == 1))
    mag = np.ldexp(n + up, q)
    largest = np.ldexp(2.0 - 2.0 ** (1 - p), emax)
    mag = np.where(mag > largest, np.inf, mag)
    return np.where(a > 0, sign * mag, hi)


def rope_store(x, positions, table, fmt):
    """The rotated keys as a store of format ``fmt`` holds them: the exact rotation of
    ``rope_apply`` rounded once to ``fmt`` (flashdreams issue, "proposed boundary":
    keys are rotated at their absolute positions before storage).  x holds values of
    ``fmt`` and the table fp32 values, so both products are exact in fp64 (at most
    24 + 24 significant bits); their difference is carried exactly as fp64 plus its
    rounding error, and rounded to ``fmt`` once.  Returns fp64 values of ``fmt``."""
    x = np.asarray(x, dtype=np.float64)
    t = np.asarray(table, dtype=np.float64)[np.asarray(positions)]      # [n, D/2, 2]
    c = t[:, None, :, 0]
    s = t[:, None, :, 1]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = round_to_format(*two_sum(x0 * c, -(x1 * s)), fmt)
    out[..., 1::2] = round_to_format(*two_sum(x0 * s, x1 * c), fmt)
    return out


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def attend(q, k, v, scale=None, causal=False, q_pos0=0, key_pos=None):
    """Naive fp64 softmax attention for one batch row.

    q: ``[n_q, H, D]``; k, v: ``[n_k, Hkv, D]`` with H a multiple of Hkv.  Query i
    sits at absolute position ``q_pos0 + i``; key j at ``key_pos[j]`` (default j).
    With ``causal`` key j is visible to query i only when its position is not later.
    Returns fp64 ``[n_q, H, D]``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, H, D = q.shape
    n_k, Hkv, _ = k.shape
    if H % Hkv:
        raise ValueError("heads must be a multiple of kv_heads")
    G = H // Hkv
    if scale is None:
        scale = default_scale(D)
    if key_pos is None:
        key_pos = np.arange(n_k)
    key_pos = np.asarray(key_pos)
    out = np.empty((n_q, H, D), dtype=np.float64)
    for h in range(H):
        kh = k[:, h // G, :]                      # [n_k, D]
        vh = v[:, h // G, :]
        s = scale * (q[:, h, :] @ kh.T)           # [n_q, n_k]
        if causal:
            qp = q_pos0 + np.arange(n_q)
            s = np.where(key_pos[None, :] <= qp[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        out[:, h, :] = (p @ vh) / p.sum(axis=1, keepdims=True)
    return out


def attend_lse(q, k, v, scale=None, causal=False, q_pos0=0):
    """``attend`` plus the natural-log log-sum-exp of each query row's scaled scores.

    Returns (out ``[n_q, H, D]``, lse ``[n_q, H]``), fp64; a row with no visible key has
    lse = -inf and output 0.  The pages' forward_with_lse (TensorRT-LLM PR "FA4
    variable-length cross-attention", Microbenchmark paragraph).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, H, D = q.shape
    n_k, Hkv, _ = k.shape
    G = H // Hkv
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((n_q, H, D), dtype=np.float64)
    lse = np.full((n_q, H), -np.inf, dtype=np.float64)
    for h in range(H):
        s = scale * (q[:, h, :] @ k[:, h // G, :].T)
        if causal:
            qp = q_pos0 + np.arange(n_q)
            s = np.where(np.arange(n_k)[None, :] <= qp[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        ok = np.isfinite(m[:, 0])
        msafe = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(s - msafe)
        tot = p.sum(axis=1, keepdims=True)
        out[ok, h, :] = ((p @ v[:, h // G, :]) / np.where(tot > 0, tot, 1.0))[ok]
        lse[ok, h] = (msafe[:, 0] + np.log(np.where(tot[:, 0] > 0, tot[:, 0], 1.0)))[ok]
    return out, lse


def merge_lse(o_a, lse_a, o_b, lse_b):
    """Combine two attentions over disjoint key sets from their outputs and LSEs:
    o = (e^lse_a o_a + e^lse_b o_b) / (e^lse_a + e^lse_b), lse = log(e^lse_a + e^lse_b).
    What forward_with_lse outputs are for (TensorRT-LLM PR "FA4 variable-length
    cross-attention", Microbenchmark paragraph); a side with lse = -inf has no keys and
    weight 0."""
    o_a, o_b = np.asarray(o_a, np.float64), np.asarray(o_b, np.float64)
    lse_a, lse_b = np.asarray(lse_a, np.float64), np.asarray(lse_b, np.float64)
    lse = np.logaddexp(lse_a, lse_b)
    safe = np.where(np.isfinite(lse), lse, 0.0)
    wa = np.where(np.isfinite(lse_a), np.exp(lse_a - safe), 0.0)[..., None]
    wb = np.where(np.isfinite(lse_b), np.exp(lse_b - safe), 0.0)[..., None]
    return wa * o_a + wb * o_b, lse


def attend_masked_full(q, k_full, v_full, kv_len, scale=None):
    """Attention over a full-capacity store with the tail ``[kv_len, cap)`` masked.

    The "before" form of the fish-speech active-prefix change: every slot is passed
    and unpopulated slots are masked out with -inf logits.
    """
    q = np.asarray(q, dtype=np.float64)
    k_full = np.asarray(k_full, dtype=np.float64)
    v_full = np.asarray(v_full, dtype=np.float64)
    n_q, H, D = q.shape
    cap, Hkv, _ = k_full.shape
    G = H // Hkv
    if scale is None:
        scale = default_scale(D)
    mask = np.arange(cap) < kv_len
    out = np.empty((n_q, H, D), dtype=np.float64)
    for h in range(H):
        s = scale * (q[:, h, :] @ k_full[:, h // G, :].T)
        s = np.where(mask[None, :], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        out[:, h, :] = (p @ v_full[:, h // G, :]) / p.sum(axis=1, keepdims=True)
    return out


def check_kv_len(kv_len: int, capacity: int) -> int:
    """Valid active prefixes are 1..capacity (fish-speech PR, regression tests, item 2)."""
    if not isinstance(kv_len, (int, np.integer)) or not 1 <= int(kv_len) <= capacity:
        raise ValueError(f"kv_len {kv_len} outside [1, {capacity}]")
    return int(kv_len)


def row_argmax(o):
    """Argmax over the last axis, lowest index on ties."""
    return np.argmax(np.asarray(o), axis=-1)


def attention_flops(n_q: int, n_k: int, heads: int, head_dim: int) -> float:
    """Algorithmic flops of one unmasked attention: 2 matmuls of 2*n_q*n_k*D each."""
    return 4.0 * n_q * n_k * heads * head_dim
