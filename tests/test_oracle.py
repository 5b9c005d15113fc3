"""Pins for the CPU fp64 oracle (no GPU).

Each test checks the oracle against something other than itself: a brute-force
simulation, a closed form, a library routine (torch SDPA in fp64) or a number the
pages print (``tests/golden/*.json``).  The last group plants plausible mistakes in
the oracle and checks that a pin catches each one.
"""
import collections
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Circular storage: brute-force ring with an explicit eviction queue
# ---------------------------------------------------------------------------
class BruteRing:
    """Physical ring simulated with a FIFO of live rolling chunks.

    Sink chunks take the first slots in order; rolling chunks take free slots in
    order until the rolling region is full, after which each new chunk takes the
    slots of the oldest live rolling chunk.  No modular arithmetic is used.
    """

    def __init__(self, sink, window, chunk):
        self.sink, self.window, self.chunk = sink, window, chunk
        self.store = [None] * window
        self.reset()

    def reset(self):
        self.n = 0
        self.live = collections.deque()     # (chunk id, first slot)
        self.where = {}                     # position -> slot, for live positions
        self.cur = None

    def reserve(self):
        c = self.n
        self.n += 1
        first_pos = c * self.chunk
        if first_pos < self.sink:
            first_slot = first_pos
        else:
            cap = (self.window - self.sink) // self.chunk
            if len(self.live) < cap:
                first_slot = self.sink + len(self.live) * self.chunk
            else:
                old, first_slot = self.live.popleft()
                for p in range(old * self.chunk, (old + 1) * self.chunk):
                    del self.where[p]
            self.live.append((c, first_slot))
        for i in range(self.chunk):
            self.where[first_pos + i] = first_slot + i
        self.cur = (first_pos, first_slot)

    def write(self, rows):
        first_pos, first_slot = self.cur
        for i, r in enumerate(rows):
            self.store[first_slot + i] = (first_pos + i, r)

    def live_positions(self):
        return sorted(self.where)


def ring_layouts():
    for chunk, sink_chunks, roll_chunks in itertools.product((1, 2, 4), range(4), range(1, 5)):
        yield chunk, sink_chunks * chunk, (sink_chunks + roll_chunks) * chunk


def test_ring_layout_count_matches_page():
    assert len(list(ring_layouts())) == golden("pages_invariants.json")["ring_layouts"]["aligned_layouts"]


def test_ring_slot_and_attended_set_match_brute_force():
    """Fill, repeated writes, wraparound and reset over 48 aligned layouts.

    Invariant of the flashdreams issue ("first experiment"): circular storage holds
    the same keys and values, in logical order, as the chronological history.
    """
    rng = np.random.default_rng(7)
    comparisons = 0
    for chunk, sink, window in ring_layouts():
        brute = BruteRing(sink, window, chunk)
        oracle = orc.ChronoCache(1, 1, 2, orc.CIRCULAR, sink=sink, window=window, chunk=chunk)
        n_chunks = sink // chunk + 2 * (window - sink) // chunk + 2   # two wraps and more
        for rnd in range(2):                                           # run, reset, run again
            for c in range(n_chunks):
                brute.reserve()
                oracle.advance()
                for rw in range(2):                                    # denoising rewrites
                    toks = rng.standard_normal((chunk, 1, 2))
                    brute.write(toks)
                    oracle.write(toks[None], -toks[None])
                    pos = oracle.attended_positions(0)
                    assert pos == brute.live_positions()
                    for p in pos:
                        s = orc.ring_slot(p, sink, window)
                        assert s == brute.where[p]
                        assert oracle.physical_slot(0, p) == s
                        bp, brow = brute.store[s]
                        assert bp == p
                        assert np.array_equal(brow, oracle.hist_k[0][p])
                        comparisons += 1
            brute.reset()
            oracle.reset()
            for s in range(window):
                brute.store[s] = None
    assert comparisons > 6912


def test_ring_fill_then_evict_oldest_tiny():
    """Tiny ring (C=4, S=4, W=16): chunks 0-3 fill, chunk 4 evicts chunk 1."""
    assert [orc.ring_slot(p, 4, 16) for p in (0, 4, 8, 12, 16, 20, 24, 28)] == [0, 4, 8, 12, 4, 8, 12, 4]
    assert orc.ring_attended(16, 4, 16) == list(range(16))
    assert orc.ring_attended(20, 4, 16) == [0, 1, 2, 3] + list(range(8, 20))


def test_ring_layout_rejects_partial_chunks():
    with pytest.raises(ValueError):
        orc.check_ring_layout(3, 16, 4)
    with pytest.raises(ValueError):
        orc.check_ring_layout(4, 14, 4)
    with pytest.raises(ValueError):
        orc.check_ring_layout(4, 4, 4)


# ---------------------------------------------------------------------------
# Attention: closed forms, invariances, a library routine
# ---------------------------------------------------------------------------
def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_single_key_returns_its_value():
    q, k, v = rnd((5, 4, 16), 1), rnd((1, 2, 16), 2), rnd((1, 2, 16), 3)
    o = orc.attend(q, k, v)
    for h in range(4):
        assert np.array_equal(o[:, h, :], np.broadcast_to(v[0, h // 2], (5, 16)))


def test_equal_keys_average_values():
    q = rnd((3, 2, 8), 4)
    k = np.broadcast_to(rnd((1, 2, 8), 5), (9, 2, 8)).copy()
    v = rnd((9, 2, 8), 6)
    o = orc.attend(q, k, v)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=0), (3, 2, 8)), atol=1e-15, rtol=0)


def test_dominant_key_selects_its_value():
    D = 8
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    k = rnd((6, 1, D), 7) * 1e-3
    k[3, 0, 0] = 1e3 * math.sqrt(D)       # logit 1e3 above the rest
    v = rnd((6, 1, D), 8)
    o = orc.attend(q, k, v)
    assert np.array_equal(o[0, 0], v[3, 0])


def test_gqa_equals_duplicated_kv_heads():
    q, k, v = rnd((7, 8, 16), 9), rnd((11, 2, 16), 10), rnd((11, 2, 16), 11)
    o_g4 = orc.attend(q, k, v)
    o_g1 = orc.attend(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1))
    assert np.array_equal(o_g4, o_g1)


def test_permutation_invariance_fp64():
    """Permuting K and V rows together leaves unmasked attention unchanged."""
    bound = golden("pages_invariants.json")["ring_layouts"]["physical_order_fp64_max_abs"]
    q, k, v = rnd((6, 4, 32), 12), rnd((40, 2, 32), 13), rnd((40, 2, 32), 14)
    o = orc.attend(q, k, v)
    worst = 0.0
    for s in range(20):
        perm = np.random.default_rng(100 + s).permutation(40)
        worst = max(worst, np.abs(orc.attend(q, k[perm], v[perm]) - o).max())
    assert worst <= 10 * bound


def sdpa_ref(q, k, v, causal=False, q_pos0=0):
    """torch SDPA in fp64 on CPU, with K/V heads expanded by repeat_interleave."""
    n_q, H, D = q.shape
    n_k, Hkv, _ = k.shape
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(H // Hkv, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(H // Hkv, dim=0)[None]
    mask = None
    if causal:
        mask = (torch.arange(n_k)[None, :] <= (q_pos0 + torch.arange(n_q))[:, None])
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n_q,n_k,H,Hkv,D", [(1, 1, 1, 1, 64), (5, 37, 4, 4, 64),
                                            (9, 130, 8, 2, 128), (16, 16, 32, 8, 128)])
def test_attend_matches_torch_sdpa(n_q, n_k, H, Hkv, D):
    q, k, v = rnd((n_q, H, D), n_q), rnd((n_k, Hkv, D), n_k), rnd((n_k, Hkv, D), n_k + 1)
    assert np.abs(orc.attend(q, k, v) - sdpa_ref(q, k, v)).max() < 1e-13


@pytest.mark.parametrize("n_q,n_k", [(7, 7), (3, 10), (1, 12)])
def test_causal_matches_torch_sdpa(n_q, n_k):
    q, k, v = rnd((n_q, 4, 32), 20), rnd((n_k, 2, 32), 21), rnd((n_k, 2, 32), 22)
    o = orc.attend(q, k, v, causal=True, q_pos0=n_k - n_q)
    assert np.abs(o - sdpa_ref(q, k, v, causal=True, q_pos0=n_k - n_q)).max() < 1e-13


def test_causal_last_query_is_unmasked():
    q, k, v = rnd((4, 2, 16), 23), rnd((9, 2, 16), 24), rnd((9, 2, 16), 25)
    oc = orc.attend(q, k, v, causal=True, q_pos0=5)
    ou = orc.attend(q[3:], k, v)
    assert np.abs(oc[3:] - ou).max() < 1e-14


# ---------------------------------------------------------------------------
# Active prefix (fish-speech PR fixture)
# ---------------------------------------------------------------------------
def test_kv_len_bounds_from_page():
    fx = golden("active_prefix_fixture.json")
    for n in fx["valid_kv_len"]:
        assert orc.check_kv_len(n, fx["capacity"]) == n
    for n in fx["invalid_kv_len"]:
        with pytest.raises(ValueError):
            orc.check_kv_len(n, fx["capacity"])


def test_prefill_decode_progression_from_page():
    fx = golden("active_prefix_fixture.json")
    cap, T = fx["capacity"], fx["prompt_len"]
    c = orc.ChronoCache(1, 2, 8, orc.LINEAR, capacity=cap)
    seen = []
    lens = []
    c.advance(n_tokens=T)
    c.write(rnd((1, T, 2, 8), 30), rnd((1, T, 2, 8), 31))
    seen.append(c.kv_len[0])
    for step in range(len(fx["progression"]) - 1):
        c.advance(n_tokens=1)
        c.write(rnd((1, 1, 2, 8), 32 + step), rnd((1, 1, 2, 8), 40 + step))
        seen.append(c.kv_len[0])
    assert seen == fx["progression"]
    # (K, V, mask) lengths at the prefill, the first decode position and the maximum prefix
    c.advance(n_tokens=cap - c.kv_len[0])
    c.write(rnd((1, cap - 5, 2, 8), 50), rnd((1, cap - 5, 2, 8), 51))
    for kv_len, want in zip(fx["observed_kvm_kv_len"], fx["observed_kvm_lengths"]):
        c.set_lengths(kv_len=[kv_len])
        k, v = c.keys_values(0)
        mask_len = len(c.attended_positions(0))
        assert [len(k), len(v), mask_len] == want
    with pytest.raises(ValueError):
        c.set_lengths(kv_len=[0])
    with pytest.raises(ValueError):
        c.set_lengths(kv_len=[cap + 1])
    with pytest.raises(ValueError):
        c.advance(n_tokens=1)


def test_active_prefix_equals_masked_full_cache():
    fx = golden("active_prefix_fixture.json")
    cap = fx["capacity"]
    k_full, v_full = rnd((cap, 2, 16), 60), rnd((cap, 2, 16), 61)
    q = rnd((2, 4, 16), 62)
    for kv_len in range(1, cap + 1):
        active = orc.attend(q, k_full[:kv_len], v_full[:kv_len])
        full = orc.attend_masked_full(q, k_full, v_full, kv_len)
        assert np.abs(active - full).max() <= fx["fp32_atol"] * 1e-6
        assert np.array_equal(orc.row_argmax(active), orc.row_argmax(full))
    # the page's fp32 bound also holds with fp32 inputs and fp32 arithmetic
    q32, k32, v32 = (x.astype(np.float32) for x in (q, k_full, v_full))
    for kv_len in (3, 4, 8):
        s = (q32[:, 0, :] @ k32[:kv_len, 0, :].T) / np.float32(4.0)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        o32 = (p @ v32[:kv_len, 0, :]) / p.sum(axis=1, keepdims=True)
        ref = orc.attend(q, k_full[:kv_len], v_full[:kv_len])[:, 0, :]
        assert np.allclose(o32, ref, rtol=fx["fp32_rtol"], atol=fx["fp32_atol"])


# ---------------------------------------------------------------------------
# Packed ragged K/V (TensorRT-LLM PR)
# ---------------------------------------------------------------------------
def test_packed_equals_padded_and_masked():
    lens = (13, 4)
    H, D, Lmax, n_q = 4, 16, 16, 5
    k = rnd((2, Lmax, H, D), 70)
    v = rnd((2, Lmax, H, D), 71)
    q = rnd((2, n_q, H, D), 72)
    cu = [0, lens[0], lens[0] + lens[1]]
    packed = orc.ChronoCache(2, H, D, orc.PACKED, capacity=cu[-1])
    packed.set_lengths(cu_seqlens=cu)
    packed.write(k, v)
    padded = orc.ChronoCache(2, H, D, orc.LINEAR, capacity=Lmax)
    padded.advance(n_tokens=Lmax)
    padded.write(k, v)
    padded.set_lengths(kv_len=list(lens))
    for b in range(2):
        kp, vp = packed.keys_values(b)
        kd, vd = padded.keys_values(b)
        assert np.array_equal(kp, kd) and np.array_equal(vp, vd)
        assert packed.physical_slot(b, 0) == cu[b]
        o = orc.attend(q[b], kp, vp)
        om = orc.attend_masked_full(q[b], k[b], v[b], lens[b])
        assert np.abs(o - om).max() < 1e-14
        # split-consistency: one branch alone gives the same result
        assert np.array_equal(o, orc.attend(q[b], k[b, :lens[b]], v[b, :lens[b]]))


def test_padded_kv_size_from_page():
    g = golden("pages_invariants.json")["cross_attention"]
    nbytes = g["cfg_branches"] * g["lkv_max"] * g["heads"] * g["head_dim"] * 2 * 2
    assert nbytes / 2**20 == g["padded_kv_bytes_mib"]


# ---------------------------------------------------------------------------
# Index write == slice assign (lingbot-world PR)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B", golden("pages_invariants.json")["index_copy"]["batches"])
def test_index_write_equals_slice_assign(B):
    n_chunks, C, cap = golden("pages_invariants.json")["index_copy"]["chunks"], 3, 32
    a = orc.ChronoCache(B, 2, 8, orc.LINEAR, capacity=cap)
    slab = np.zeros((B, cap, 2, 8))
    for c in range(n_chunks):
        k, v = rnd((B, C, 2, 8), 80 + c), rnd((B, C, 2, 8), 90 + c)
        a.write(k, v, slots=list(range(c * C, (c + 1) * C)))
        slab[:, c * C:(c + 1) * C] = k
        a.set_lengths(kv_len=[(c + 1) * C] * B)
        for b in range(B):
            kk, _ = a.keys_values(b)
            assert np.array_equal(kk, slab[b, :(c + 1) * C])


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by one of the pins above
# ---------------------------------------------------------------------------
def test_planted_ring_slot_off_by_one_is_caught(monkeypatch):
    real = orc.ring_slot
    monkeypatch.setattr(orc, "ring_slot", lambda p, s, w: real(p + (p >= s), s, w))
    with pytest.raises(AssertionError):
        test_ring_slot_and_attended_set_match_brute_force()


def test_planted_attended_set_error_is_caught(monkeypatch):
    real = orc.ring_attended
    monkeypatch.setattr(orc, "ring_attended", lambda e, s, w: real(e, s, w + 1))
    with pytest.raises(AssertionError):
        test_ring_slot_and_attended_set_match_brute_force()


def test_planted_scale_error_is_caught(monkeypatch):
    monkeypatch.setattr(orc, "default_scale", lambda d: 1.0 / d)
    with pytest.raises(AssertionError):
        test_attend_matches_torch_sdpa(5, 37, 4, 4, 64)


def test_planted_gqa_mapping_is_caught():
    """A mod-instead-of-divide head mapping differs from repeat_interleave."""
    q, k, v = rnd((3, 8, 16), 9), rnd((5, 2, 16), 10), rnd((5, 2, 16), 11)
    good = orc.attend(q, k, v)
    wrong = orc.attend(q, np.repeat(k, 4, axis=1)[:, [h % 2 for h in range(8)]],
                       np.repeat(v, 4, axis=1)[:, [h % 2 for h in range(8)]])
    assert np.abs(good - sdpa_ref(q, k, v)).max() < 1e-13
    assert np.abs(wrong - sdpa_ref(q, k, v)).max() > 1e-3


# ---------------------------------------------------------------------------
# RoPE at absolute positions
# ---------------------------------------------------------------------------
def test_rope_apply_matches_independent_rotation():
    from diffusion_serving_gb300 import workloads as wl
    D, n = 64, 9
    table = wl.rope_table(100, D)
    x = torch.randn(1, n, 2, D, dtype=torch.float64)
    pos = [0, 1, 5, 17, 33, 50, 64, 80, 99]
    ref = wl.rope_rotate(x, pos)[0].numpy()            # computes its own fp64 cos/sin
    got = orc.rope_apply(x[0].numpy(), pos, table.numpy())
    assert np.abs(got - ref).max() < 1e-5              # the table is fp32-rounded


def test_rope_apply_invariants():
    from diffusion_serving_gb300 import workloads as wl
    D = 128
    table = wl.rope_table(4096, D).numpy().astype(np.float64)
    x = rnd((6, 3, D), 90)
    pos = [0, 1, 7, 1000, 4000, 4095]
    y = orc.rope_apply(x, pos, table)
    # position 0 is the identity
    assert np.array_equal(y[0], x[0])
    # each pair keeps its norm (cos^2 + sin^2 = 1 up to the table's fp32 rounding)
    n_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.abs(n_y - n_x).max() <= 1e-6 * n_x.max()
    # turning back by the conjugate angle restores x
    conj = table.copy()
    conj[..., 1] = -conj[..., 1]
    assert np.abs(orc.rope_apply(y, pos, conj) - x).max() < 1e-6


def test_planted_rope_sign_error_is_caught(monkeypatch):
    real = orc.rope_apply

    def wrong(x, positions, table):
        t = np.array(table, copy=True)
        t[..., 1] = -t[..., 1]
        return real(x, positions, t)
    monkeypatch.setattr(orc, "rope_apply", wrong)
    with pytest.raises(AssertionError):
        test_rope_apply_matches_independent_rotation()


# ---------------------------------------------------------------------------
# Log-sum-exp output and the merge of partial attentions
# ---------------------------------------------------------------------------
def test_lse_matches_torch_logsumexp_and_attend():
    q, k, v = rnd((7, 4, 32), 200), rnd((50, 2, 32), 201), rnd((50, 2, 32), 202)
    o, lse = orc.attend_lse(q, k, v)
    assert np.abs(o - orc.attend(q, k, v)).max() < 1e-14
    scale = 1 / math.sqrt(32)
    for h in range(4):
        s = torch.from_numpy(scale * (q[:, h, :] @ k[:, h // 2, :].T))
        assert np.abs(lse[:, h] - torch.logsumexp(s, dim=1).numpy()).max() < 1e-12


def test_lse_closed_forms():
    q, k, v = rnd((3, 2, 16), 203), rnd((1, 2, 16), 204), rnd((1, 2, 16), 205)
    _, lse = orc.attend_lse(q, k, v)
    for h in range(2):
        assert np.allclose(lse[:, h], (q[:, h, :] @ k[0, h]) / 4.0, atol=1e-14, rtol=0)
    kk = np.broadcast_to(k, (9, 2, 16)).copy()
    _, lse9 = orc.attend_lse(q, kk, rnd((9, 2, 16), 206))
    assert np.allclose(lse9, lse + math.log(9), atol=1e-13, rtol=0)


def test_merge_of_halves_equals_attention_over_union():
    q, k, v = rnd((6, 4, 32), 210), rnd((40, 2, 32), 211), rnd((40, 2, 32), 212)
    o, lse = orc.attend_lse(q, k, v)
    oa, la = orc.attend_lse(q, k[:17], v[:17])
    ob, lb = orc.attend_lse(q, k[17:], v[17:])
    om, lm = orc.merge_lse(oa, la, ob, lb)
    assert np.abs(om - o).max() < 1e-13 and np.abs(lm - lse).max() < 1e-13


def test_causal_lse_of_row_without_keys():
    q, k, v = rnd((4, 2, 8), 220), rnd((2, 2, 8), 221), rnd((2, 2, 8), 222)
    o, lse = orc.attend_lse(q, k, v, causal=True, q_pos0=-2)       # rows 0, 1 see nothing
    assert np.all(np.isneginf(lse[:2])) and np.all(o[:2] == 0)
    assert np.all(np.isfinite(lse[2:]))


def test_roll_left_matches_brute_force_deque():
    """The chronological store after a roll holds the sink, then the retained tokens in
    order (a deque that drops its oldest rolling chunk)."""
    S, W, C = 2, 10, 2
    store = np.arange(3 * W).reshape(3, W)
    out = orc.roll_left(store, S, W, C)
    for b in range(3):
        rolling = collections.deque(store[b, S:W].tolist())
        for _ in range(C):
            rolling.popleft()
        assert out[b, :S].tolist() == store[b, :S].tolist()
        assert out[b, S:W - C].tolist() == list(rolling)
        assert out[b, W - C:].tolist() == store[b, W - C:].tolist()


# ---------------------------------------------------------------------------
# What a store holds after the fused rotation: the exact rotation rounded once
# ---------------------------------------------------------------------------
def round_exact(D, fmt):
    """Nearest value of ``fmt`` to the rational D, ties to the even significand, by
    exact rational arithmetic (the textbook definition, independent of fp64)."""
    from fractions import Fraction as Fr
    p, emin, emax = orc.FORMATS[fmt]
    if D == 0:
        return 0.0
    sign = -1 if D < 0 else 1
    a = abs(D)
    E = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** E > a:
        E -= 1
    while Fr(2) ** (E + 1) <= a:
        E += 1
    u = Fr(2) ** (max(E, emin) - (p - 1))
    below = math.floor(a / u)
    lo_v, hi_v = below * u, (below + 1) * u
    if a - lo_v < hi_v - a or (a - lo_v == hi_v - a and below % 2 == 0):
        v = lo_v
    else:
        v = hi_v
    if v > (2 - Fr(2) ** (1 - p)) * Fr(2) ** emax:
        return sign * math.inf
    return sign * float(v)


def exact_rotation(x0, x1, c, s):
    from fractions import Fraction as Fr
    return (Fr(x0) * Fr(c) - Fr(x1) * Fr(s), Fr(x0) * Fr(s) + Fr(x1) * Fr(c))


def as_fmt(a, fmt):
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[fmt]
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(dt).double().numpy()


def rope_cases(fmt, n, seed):
    """Pairs (x0, x1) of ``fmt`` and fp32 (cos, sin) entries: random magnitudes over
    many binades, plus constructed ties (the exact product on a midpoint of ``fmt``)
    and near-ties (a tiny second product pushing it just off), results in the
    subnormal range and past the largest finite value."""
    rng = np.random.default_rng(seed)
    p, emin, emax = orc.FORMATS[fmt]
    top = {"bf16": 100, "f16": 14, "f32": 100}[fmt]
    x = as_fmt(rng.standard_normal((n, 2)) * np.exp2(rng.integers(-20, top, (n, 2))), fmt)
    cs = rng.uniform(-1, 1, (n, 2)).astype(np.float32).astype(np.float64)
    cs[::7, 1] = np.float32(rng.uniform(-1, 1, len(cs[::7])) * 2.0 ** -30)
    # ties and near-ties: x0 = 1, cos = a midpoint of fmt (p + 1 significant bits),
    # x1 * sin = 0, or +-(a 24-bit value) x 2^-60: below half an fp64 ulp of the
    # midpoint, so the fp64 difference lands on the midpoint and only the exact rest
    # tells the side
    k = n // 4
    mid = (2 ** p + 2 * rng.integers(0, 2 ** (p - 1), k) + 1) / 2.0 ** (p + 1)
    x[:k, 0] = 1.0
    cs[:k, 0] = mid
    x[:k, 1] = as_fmt(np.where(np.arange(k) % 3 == 0, 0.0, 1.0), fmt)
    tiny = np.float32(rng.uniform(1, 2, k)).astype(np.float64) * 2.0 ** -60
    cs[:k, 1] = np.where(np.arange(k) % 3 == 1, tiny, -tiny)
    if fmt == "f16":                       # subnormal results and overflow
        x[k:k + 8] = [[6.1e-5, 3.0e-5]] * 8
        x[k + 8:k + 12] = [[65504.0, -65504.0]] * 4
        cs[k + 8:k + 12] = [[0.75, 0.75]] * 4
    return x, cs


@pytest.mark.parametrize("fmt", ["bf16", "f16", "f32"])
def test_rope_store_is_the_exact_rotation_rounded_once(fmt):
    x, cs = rope_cases(fmt, 1200, {"bf16": 1, "f16": 2, "f32": 3}[fmt])
    n = len(x)
    table = cs.reshape(n, 1, 2)                       # one pair per position
    got = orc.rope_store(x.reshape(n, 1, 2), np.arange(n), table, fmt).reshape(n, 2)
    from fractions import Fraction as Fr
    inexact = 0
    for i in range(n):
        a, b = exact_rotation(x[i, 0], x[i, 1], cs[i, 0], cs[i, 1])
        want = (round_exact(a, fmt), round_exact(b, fmt))
        assert got[i, 0] == want[0] and got[i, 1] == want[1], (i, x[i], cs[i], got[i], want)
        inexact += Fr(float(a)) != a
    # the rotation differs from its fp64 rounding in some of these cases (or the pin
    # would not exercise the carried remainder)
    assert inexact > 0


def test_rope_store_matches_numpy_rounding_where_fp64_is_exact():
    """With both products of one binade the fp64 rotation is exact, and NumPy's own
    fp64 -> fp16 / fp32 conversion (correctly rounded) must agree."""
    from diffusion_serving_gb300 import workloads as wl
    D = 64
    table = wl.rope_table(512, D).numpy()
    x16 = rnd((40, 2, D), 300).astype(np.float16).astype(np.float64)
    pos = np.arange(3, 43) * 11
    ref = orc.rope_apply(x16, pos, table)
    assert np.array_equal(orc.rope_store(x16, pos, table, "f16"),
                          ref.astype(np.float16).astype(np.float64))
    x32 = rnd((40, 2, D), 301).astype(np.float32).astype(np.float64)
    lo_free = orc.rope_store(x32, pos, table, "f32")
    want = orc.rope_apply(x32, pos, table).astype(np.float32).astype(np.float64)
    # fp32 inputs: the products have 48 bits, so fp64 rounds some differences; those
    # may differ from NumPy's conversion only where fp64 landed on an fp32 midpoint
    assert np.mean(lo_free == want) > 0.999


def test_planted_double_rounding_is_caught(monkeypatch):
    """Rounding the fp64 rotation to the format (two roundings) instead of the exact
    rotation fails the exact pin on the near-tie cases."""
    real = orc.round_to_format

    def twice(hi, lo, fmt):
        return real(hi, np.zeros_like(np.asarray(hi, dtype=np.float64)), fmt)
    monkeypatch.setattr(orc, "round_to_format", twice)
    with pytest.raises(AssertionError):
        test_rope_store_is_the_exact_rotation_rounded_once("bf16")
