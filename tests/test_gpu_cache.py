"""GPU tests of slot reservation, writes, lengths and device-side error reporting.

The cache contents must be bit-exact against the oracle's chronological history read
through its closed-form slot map (flashdreams issue "add an opt-in circular KV
policy for streaming attention", "first experiment"), and a device-index write must
equal torch slice-assignment (lingbot-world PR "refactor(kv): index_copy_ for
KV-cache writes", "Verification").
"""
import numpy as np
import pytest
import torch

from oracle import kvc_oracle as orc
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from diffusion_serving_gb300 import kvc


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def store_matches_history(cache, oracle, b, dtype):
    """Every attended position of row b sits, bit-exact, at its closed-form slot."""
    pos = oracle.attended_positions(b)
    slots = torch.tensor([oracle.physical_slot(b, p) for p in pos], device="cuda")
    for store, hist in ((cache.k_store, oracle.hist_k[b]), (cache.v_store, oracle.hist_v[b])):
        want = torch.from_numpy(np.stack([hist[p] for p in pos])).to(dtype)
        got = store[b].index_select(0, slots).cpu()
        if not torch.equal(bits(got), bits(want)):
            return False
    return True


@pytest.mark.parametrize("chunk,sink_c,roll_c", [(4, 1, 3), (2, 0, 4), (1, 3, 2), (4, 2, 1)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ring_fill_rewrite_wrap_reset_bit_exact(chunk, sink_c, roll_c, dtype):
    B, Hkv, D = 2, 2, 64
    sink, window = sink_c * chunk, (sink_c + roll_c) * chunk
    cache = kvc.KVCache(B, Hkv, Hkv, D, dtype, "circular", sink=sink, window=window, chunk=chunk)
    oracle = orc.ChronoCache(B, Hkv, D, orc.CIRCULAR, sink=sink, window=window, chunk=chunk)
    g = torch.Generator().manual_seed(5)
    n_chunks = sink_c + 2 * roll_c + 2
    for rnd in range(2):
        for c in range(n_chunks):
            cache.advance()
            oracle.advance()
            for rw in range(2):
                k = torch.randn(B, chunk, Hkv, D, generator=g).to(dtype)
                v = torch.randn(B, chunk, Hkv, D, generator=g).to(dtype)
                cache.write(k.cuda(), v.cuda())
                oracle.write(k.double().numpy(), v.double().numpy())
                for b in range(B):
                    assert store_matches_history(cache, oracle, b, dtype)
                state = cache.row_state()
                for b in range(B):
                    assert state[b][3] == len(oracle.attended_positions(b))
        cache.reset()
        oracle.reset()
        assert all(r == [0, 0, 0, 0] for r in cache.row_state())
    assert cache.get_error() == 0


@pytest.mark.parametrize("B", [1, 2])
def test_index_write_equals_slice_assign(B):
    """Writes at a device index tensor equal slice-assignment, 7 chunks."""
    H, D, C, cap = 4, 128, 5, 64
    cache = kvc.KVCache(B, H, H, D, torch.bfloat16, "linear", capacity=cap)
    ref_k = torch.zeros(B, cap, H, D, dtype=torch.bfloat16, device="cuda")
    ref_v = torch.zeros_like(ref_k)
    cache.k_store.zero_()
    cache.v_store.zero_()
    idx = torch.empty(C, dtype=torch.int32, device="cuda")
    for c in range(7):
        k = torch.randn(B, C, H, D, device="cuda").to(torch.bfloat16)
        v = torch.randn(B, C, H, D, device="cuda").to(torch.bfloat16)
        idx.copy_(torch.arange(c * C, (c + 1) * C, dtype=torch.int32))
        cache.write(k, v, slots=idx)
        ref_k[:, c * C:(c + 1) * C] = k
        ref_v[:, c * C:(c + 1) * C] = v
        assert torch.equal(bits(cache.k_store), bits(ref_k))
        assert torch.equal(bits(cache.v_store), bits(ref_v))
    assert cache.get_error() == 0


def test_linear_advance_progression_and_overflow():
    """kv_len follows prefill T then T+1, T+2 ...; advancing past capacity is reported."""
    cache = kvc.KVCache(1, 2, 2, 64, torch.float16, "linear", capacity=8)
    cache.advance(n_tokens=3)
    seen = [cache.row_state()[0][3]]
    for _ in range(2):
        cache.advance(n_tokens=1)
        seen.append(cache.row_state()[0][3])
    assert seen == [3, 4, 5]
    cache.advance(n_tokens=3)
    assert cache.row_state()[0][3] == 8
    assert cache.get_error() == 0
    cache.advance(n_tokens=1)
    assert cache.get_error() == kvc.DEV_OVERFLOW
    assert cache.row_state()[0][3] == 8


def test_kv_len_bounds_on_device():
    """kv_len 1 and capacity are accepted, 0 and capacity + 1 rejected."""
    cache = kvc.KVCache(1, 2, 2, 64, torch.float16, "linear", capacity=8)
    for n, ok in ((1, True), (8, True), (0, False), (9, False)):
        cache.set_lengths(kv_len=torch.tensor([n], dtype=torch.int32, device="cuda"))
        err = cache.get_error()
        assert (err == 0) == ok, (n, err)
    with pytest.raises(kvc.KvcError):
        cache.advance(n_tokens=9)


def test_bad_slots_and_cu_seqlens_are_reported_not_faulted():
    cache = kvc.KVCache(2, 2, 2, 64, torch.bfloat16, "linear", capacity=16)
    before = cache.k_store.clone()
    k = torch.randn(2, 3, 2, 64, device="cuda").to(torch.bfloat16)
    cache.write(k, k, slots=torch.tensor([0, 16, -1], dtype=torch.int32, device="cuda"))
    assert cache.get_error() == kvc.DEV_BAD_SLOT
    assert torch.equal(bits(cache.k_store[:, 0]), bits(k[:, 0]))
    assert torch.equal(bits(cache.k_store[:, 1:]), bits(before[:, 1:]))
    # write before any reservation
    cache.write(k, k)
    assert cache.get_error() == kvc.DEV_NO_CHUNK
    # attend with kv_len 0 leaves the output untouched and reports
    q = torch.randn(2, 4, 2, 64, device="cuda").to(torch.bfloat16)
    out = torch.full_like(q, 7.0)
    cache.attend(q, out)
    assert cache.get_error() & kvc.DEV_BAD_KVLEN
    assert torch.all(out == 7.0)
    packed = kvc.KVCache(2, 2, 2, 64, torch.bfloat16, "packed", capacity=16)
    for cu in ([0, 5, 4], [1, 3, 5], [0, 8, 17], [0, 0, 3]):
        packed.set_lengths(cu_seqlens=torch.tensor(cu, dtype=torch.int32, device="cuda"))
        assert packed.get_error() == kvc.DEV_BAD_CUSEQ, cu


def test_host_validation():
    with pytest.raises(kvc.KvcError):
        kvc.KVCache(1, 3, 2, 64, torch.float16, "linear", capacity=8)          # H % Hkv
    with pytest.raises(kvc.KvcError):
        kvc.KVCache(1, 2, 2, 64, torch.float16, "circular", sink=3, window=16, chunk=4)
    ring = kvc.KVCache(1, 2, 2, 64, torch.float16, "circular", sink=4, window=16, chunk=4)
    q = torch.randn(1, 4, 2, 64, device="cuda").half()
    with pytest.raises(kvc.KvcError) as e:
        ring.attend(q, flags=kvc.CAUSAL)
    assert e.value.code == kvc.ERR_UNSUPPORTED
    with pytest.raises(kvc.KvcError):
        ring.advance(n_tokens=3)
    with pytest.raises(kvc.KvcError):
        ring.write(q[:, :3, :, :], q[:, :3, :, :])
    # shapes, dtypes and strides the binding refuses before any call
    lin = kvc.KVCache(2, 4, 2, 64, torch.bfloat16, "linear", capacity=32)
    lin.advance(n_tokens=8)
    k = torch.randn(2, 8, 2, 64, device="cuda").bfloat16()
    for bad_k in (k.half(), k[:, :, :1].contiguous(), torch.randn(2, 8, 4, 64, device="cuda").bfloat16()):
        with pytest.raises(ValueError):
            lin.write(bad_k, bad_k)
    with pytest.raises(ValueError):
        lin.write(k, k[:, :4].contiguous())
    qq = torch.randn(2, 5, 4, 64, device="cuda").bfloat16()
    for bad_q in (qq.half(), qq[:1].contiguous(), torch.randn(2, 5, 2, 64, device="cuda").bfloat16()):
        with pytest.raises(ValueError):
            lin.attend(bad_q)
    with pytest.raises(ValueError):
        lin.attend(torch.randn(2, 4, 5, 64, device="cuda").bfloat16().transpose(1, 2))
    with pytest.raises(ValueError):
        lin.attend(qq, torch.empty(2, 5, 4, 64, device="cuda", dtype=torch.float16))
    # empty calls are argument errors at the C boundary (kvc.h conventions)
    out = torch.full_like(qq, 3.0)
    for call in (lambda: kvc.kvc_attend(lin.handle, qq, out, 0),
                 lambda: kvc.kvc_write(lin.handle, k, k, 0),
                 lambda: kvc.kvc_merge(torch.bfloat16, 0, 64, qq, qq, qq, qq, out)):
        with pytest.raises(kvc.KvcError) as e:
            call()
        assert e.value.code == kvc.ERR_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    assert lin.get_error() == 0


def test_graph_replay_writes_the_device_slot():
    """A captured advance+write+attend replayed per chunk equals the eager run and
    writes a different slot each chunk (flashdreams issue, "proposed boundary")."""
    B, H, D, C, S, W = 2, 4, 128, 8, 8, 40
    n_chunks = 9
    ins = [tuple(torch.randn(B, C, H, D, device="cuda").to(torch.bfloat16) for _ in range(3))
           for _ in range(n_chunks)]
    eager = kvc.KVCache(B, H, H, D, torch.bfloat16, "circular", sink=S, window=W, chunk=C)
    eager_out = []
    for q, k, v in ins:
        eager.advance()
        eager.write(k, v)
        eager_out.append(eager.attend(q))
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        cache = kvc.KVCache(B, H, H, D, torch.bfloat16, "circular", sink=S, window=W, chunk=C)
        qb, kb, vb = (torch.empty_like(x) for x in ins[0])
        ob = torch.empty_like(qb)
        # warm-up outside capture: chunk 0
        qb.copy_(ins[0][0]); kb.copy_(ins[0][1]); vb.copy_(ins[0][2])
        cache.advance(stream=side)
        cache.write(kb, vb, stream=side)
        cache.attend(qb, ob, stream=side)
    side.synchronize()
    outs = [ob.clone()]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        cache.advance(stream=side)
        cache.write(kb, vb, stream=side)
        cache.attend(qb, ob, stream=side)
    bases = []
    for c in range(1, n_chunks):
        qb.copy_(ins[c][0]); kb.copy_(ins[c][1]); vb.copy_(ins[c][2])
        graph.replay()
        torch.cuda.synchronize()
        outs.append(ob.clone())
        bases.append(cache.row_state()[0][1])
    for a, b in zip(outs, eager_out):
        assert torch.equal(bits(a), bits(b))
    # every slot was written by now: the stores agree bit for bit
    assert torch.equal(bits(cache.k_store), bits(eager.k_store))
    assert torch.equal(bits(cache.v_store), bits(eager.v_store))
    assert bases == [8, 16, 24, 32, 8, 16, 24, 32]
    assert cache.get_error() == 0 and eager.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_roll_comparator_matches_chronological_copy(dtype):
    """The comparator copy (what the circular layout avoids) moves the retained rolling
    tokens one chunk to the left, bit for bit."""
    B, Hkv, D, C, S, W = 3, 2, 64, 4, 8, 40
    cache = kvc.KVCache(B, Hkv, Hkv, D, dtype, "circular", sink=S, window=W, chunk=C)
    cache.k_store.normal_()
    cache.v_store.normal_()
    before_k, before_v = cache.k_store.cpu(), cache.v_store.cpu()
    scratch = torch.empty(kvc.kvc_roll_scratch_bytes(cache.cfg), dtype=torch.uint8, device="cuda")
    kvc.kvc_roll_window(cache.handle, scratch)
    torch.cuda.synchronize()
    want_k = orc.roll_left(bits(before_k).numpy(), S, W, C)
    want_v = orc.roll_left(bits(before_v).numpy(), S, W, C)
    assert np.array_equal(bits(cache.k_store.cpu()).numpy(), want_k)
    assert np.array_equal(bits(cache.v_store.cpu()).numpy(), want_v)


@pytest.mark.parametrize("n", [1, 3, 30, 300])
def test_append_equals_advance_then_write(n):
    """kvc_append (one launch for a decode step's few tokens, the advance + write pair
    for appends of more than 128 KiB) leaves the same store bytes and row state as kvc_advance followed by
    kvc_write."""
    B, Hkv, D, cap = 2, 8, 128, 1024
    a = kvc.KVCache(B, 32, Hkv, D, torch.float16, "linear", capacity=cap)
    w = kvc.KVCache(B, 32, Hkv, D, torch.float16, "linear", capacity=cap)
    for c in (a, w):
        c.k_store.zero_()
        c.v_store.zero_()
    g = torch.Generator(device="cuda").manual_seed(n)
    for step in range(3):
        k = torch.randn(B, n, Hkv, D, device="cuda", generator=g).half()
        v = torch.randn(B, n, Hkv, D, device="cuda", generator=g).half()
        a.append(k, v)
        w.advance(n_tokens=n)
        w.write(k, v)
        assert a.row_state() == w.row_state()
    assert torch.equal(bits(a.k_store), bits(w.k_store)) and torch.equal(bits(a.v_store), bits(w.v_store))
    assert a.row_state()[0] == [3, 2 * n, 3 * n, 3 * n]
    assert a.get_error() == 0 and w.get_error() == 0


def test_append_past_capacity_is_reported_and_skipped():
    cap = 8
    c = kvc.KVCache(1, 2, 2, 64, torch.bfloat16, "linear", capacity=cap)
    k = torch.randn(1, 3, 2, 64, device="cuda").bfloat16()
    c.append(k, k)
    c.append(k, k)
    before = c.row_state()
    c.append(k, k)                                   # 6 + 3 > 8
    assert c.get_error() == kvc.DEV_OVERFLOW
    assert c.row_state() == before
    ring = kvc.KVCache(1, 2, 2, 64, torch.bfloat16, "circular", sink=4, window=16, chunk=4)
    with pytest.raises(kvc.KvcError) as e:
        ring.append(k[:, :1].contiguous(), k[:, :1].contiguous())
    assert e.value.code == kvc.ERR_UNSUPPORTED


def test_captured_append_attend_decode_steps_match_the_oracle():
    """A decode step (append the token's K/V, attend) captured once and replayed: each
    replay appends at the next slot and attends the whole prefix (fish-speech PR, "Change")."""
    B, H, Hkv, D, cap, T = 1, 32, 8, 128, 4096, 234
    c = kvc.KVCache(B, H, Hkv, D, torch.float16, "linear", capacity=cap)
    orc_c = orc.ChronoCache(B, Hkv, D, orc.LINEAR, capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(77)
    kp = torch.randn(B, T, Hkv, D, device="cuda", generator=g).half()
    vp = torch.randn(B, T, Hkv, D, device="cuda", generator=g).half()
    c.append(kp, vp)
    orc_c.advance(n_tokens=T)
    orc_c.write(to64(kp), to64(vp))
    k1 = torch.empty(B, 1, Hkv, D, device="cuda").half()
    v1 = torch.empty_like(k1)
    q1 = torch.empty(B, 1, H, D, device="cuda").half()
    o1 = torch.empty_like(q1)
    q1.zero_()
    c.attend(q1, o1)                                 # the decode kernel's first launch, outside capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        c.append(k1, v1, stream=side)
        c.attend(q1, o1, stream=side)
    for i in range(20):
        for t in (k1, v1, q1):
            t.normal_(generator=g)
        graph.replay()
        torch.cuda.synchronize()
        orc_c.advance(n_tokens=1)
        orc_c.write(to64(k1), to64(v1))
        kk, vv = orc_c.keys_values(0)
        assert kk.shape[0] == T + i + 1
        assert_close(o1[0], orc.attend(to64(q1[0]), kk, vv), f"step {i}")
    assert c.row_state()[0][3] == T + 20
    assert c.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("prefix", [0, 5, 111, 112, 447, 448, 449, 490, 560, 561, 672, 673, 2500])
def test_fused_append_attend_equals_append_then_attend(dtype, prefix):
    """kvc_append_attend_decode leaves the same store bytes and row state as kvc_append
    followed by kvc_attend, and its output, like theirs, matches the oracle over the prefix
    plus the new token, for prefixes streamed by one block (up to 448 slots: 4 tiles of
    112) or split (449 and longer), on and beside tile edges and the block-count
    threshold, over three consecutive steps with rows of different lengths."""
    B, H, Hkv, D, cap = 2, 32, 8, 128, 4096
    fused = kvc.KVCache(B, H, Hkv, D, dtype, "linear", capacity=cap)
    ref = kvc.KVCache(B, H, Hkv, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(prefix + 3)
    for c in (fused, ref):
        c.k_store.zero_()
        c.v_store.zero_()
    lens = [prefix, max(prefix - 3, 0) + (7 if prefix else 0)]
    hist_k, hist_v = [], []
    for b in range(B):
        kp = torch.randn(1, lens[b], Hkv, D, device="cuda", generator=g).to(dtype)
        vp = torch.randn(1, lens[b], Hkv, D, device="cuda", generator=g).to(dtype)
        hist_k.append(kp[0])
        hist_v.append(vp[0])
        for c in (fused, ref):
            c.k_store[b, :lens[b]] = kp[0]
            c.v_store[b, :lens[b]] = vp[0]
            meta = c.meta.view(torch.int32)
            row = 4 + 4 * b
            meta[row:row + 4] = torch.tensor([1 if lens[b] else 0, 0, lens[b], lens[b]], dtype=torch.int32)
    for step in range(3):
        k = torch.randn(B, 1, Hkv, D, device="cuda", generator=g).to(dtype)
        v = torch.randn(B, 1, Hkv, D, device="cuda", generator=g).to(dtype)
        q = torch.randn(B, 1, H, D, device="cuda", generator=g).to(dtype)
        out = torch.full_like(q, float("nan"))
        fused.append_attend(k, v, q, out)
        ref.append(k, v)
        want = ref.attend(q)
        torch.cuda.synchronize()
        assert fused.row_state() == ref.row_state(), f"step {step}"
        for b in range(B):
            hist_k[b] = torch.cat([hist_k[b], k[b]])
            hist_v[b] = torch.cat([hist_v[b], v[b]])
            o = orc.attend(to64(q[b]), to64(hist_k[b]), to64(hist_v[b]))
            assert_close(out[b], o, f"step {step} row {b} vs oracle")
            # the two-launch step's output is checked against the same oracle: both are
            # within the tolerance of it, the fused one without the 16-bit P of the new key
            assert_close(want[b], o, f"step {step} row {b}, append + attend vs oracle")
    assert torch.equal(bits(fused.k_store), bits(ref.k_store)) and torch.equal(bits(fused.v_store), bits(ref.v_store))
    assert fused.get_error() == 0 and ref.get_error() == 0


def test_fused_append_attend_past_capacity_and_unsupported():
    B, H, Hkv, D, cap = 1, 8, 2, 64, 4
    c = kvc.KVCache(B, H, Hkv, D, torch.float16, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(5)
    for _ in range(cap):
        k = torch.randn(B, 1, Hkv, D, device="cuda", generator=g).half()
        q = torch.randn(B, 1, H, D, device="cuda", generator=g).half()
        c.append_attend(k, k, q)
    assert c.get_error() == 0
    before = c.row_state()
    c.append_attend(k, k, q)                             # slot cap is past the store
    assert c.get_error() == kvc.DEV_OVERFLOW
    assert c.row_state() == before
    ring = kvc.KVCache(1, 8, 2, 64, torch.float16, "circular", sink=4, window=16, chunk=4)
    with pytest.raises(kvc.KvcError) as e:
        ring.append_attend(k, k, q)
    assert e.value.code == kvc.ERR_UNSUPPORTED


def test_captured_fused_decode_steps_match_the_oracle():
    """The fused step captured once and replayed: each replay appends at the next slot
    and attends the prefix up to it, as the two-launch step does."""
    B, H, Hkv, D, cap, T = 1, 32, 8, 128, 4096, 234
    c = kvc.KVCache(B, H, Hkv, D, torch.float16, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(78)
    kp = torch.randn(B, T, Hkv, D, device="cuda", generator=g).half()
    vp = torch.randn(B, T, Hkv, D, device="cuda", generator=g).half()
    c.append(kp, vp)
    hk, hv = kp[0], vp[0]
    k1 = torch.zeros(B, 1, Hkv, D, device="cuda").half()
    v1 = torch.zeros_like(k1)
    q1 = torch.zeros(B, 1, H, D, device="cuda").half()
    o1 = torch.empty_like(q1)
    warm = kvc.KVCache(B, H, Hkv, D, torch.float16, "linear", capacity=cap)
    warm.append_attend(k1, v1, q1)                   # the kernel's first launch, outside capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        c.append_attend(k1, v1, q1, o1, stream=side)
    torch.cuda.synchronize()
    assert c.row_state()[0][2] == T                  # capture ran nothing
    for step in range(4):
        k1.copy_(torch.randn(B, 1, Hkv, D, device="cuda", generator=g).half())
        v1.copy_(torch.randn(B, 1, Hkv, D, device="cuda", generator=g).half())
        q1.copy_(torch.randn(B, 1, H, D, device="cuda", generator=g).half())
        graph.replay()
        torch.cuda.synchronize()
        hk = torch.cat([hk, k1[0]])
        hv = torch.cat([hv, v1[0]])
        assert_close(o1[0], orc.attend(to64(q1[0]), to64(hk), to64(hv)), f"replay {step}")
    assert c.row_state()[0][2] == T + 4
    assert torch.equal(bits(c.k_store[0, :T + 4]), bits(hk)) and torch.equal(bits(c.v_store[0, :T + 4]), bits(hv))
    assert c.get_error() == 0


@pytest.mark.parametrize("heads,kv_heads,head_dim", [(8, 8, 64), (64, 8, 128), (16, 8, 64)])
def test_fused_append_attend_other_head_shapes(heads, kv_heads, head_dim):
    """The append instantiation for one q head per kv head, eight per kv head and
    head_dim 64: the same store and row state as append + attend, output against the
    oracle, with one row on one block and one split over several."""
    B, cap = 2, 2048
    dtype = torch.bfloat16
    fused = kvc.KVCache(B, heads, kv_heads, head_dim, dtype, "linear", capacity=cap)
    ref = kvc.KVCache(B, heads, kv_heads, head_dim, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(heads + head_dim)
    for c in (fused, ref):               # past the prefixes both stores hold the same bytes
        c.k_store.zero_()
        c.v_store.zero_()
    lens = (300, 1500)
    for b, n in enumerate(lens):
        kp = torch.randn(n, kv_heads, head_dim, device="cuda", generator=g).to(dtype)
        vp = torch.randn(n, kv_heads, head_dim, device="cuda", generator=g).to(dtype)
        for c in (fused, ref):
            c.k_store[b, :n] = kp
            c.v_store[b, :n] = vp
            row = 4 + 4 * b
            c.meta[row:row + 4] = torch.tensor([1, 0, n, n], dtype=torch.int32)
    k = torch.randn(B, 1, kv_heads, head_dim, device="cuda", generator=g).to(dtype)
    v = torch.randn(B, 1, kv_heads, head_dim, device="cuda", generator=g).to(dtype)
    q = torch.randn(B, 1, heads, head_dim, device="cuda", generator=g).to(dtype)
    out = fused.append_attend(k, v, q)
    ref.append(k, v)
    torch.cuda.synchronize()
    assert fused.row_state() == ref.row_state()
    assert torch.equal(bits(fused.k_store), bits(ref.k_store)) and torch.equal(bits(fused.v_store), bits(ref.v_store))
    for b, n in enumerate(lens):
        o = orc.attend(to64(q[b]), to64(fused.k_store[b, :n + 1]), to64(fused.v_store[b, :n + 1]))
        assert_close(out[b], o, f"row {b}")
    assert fused.get_error() == 0
