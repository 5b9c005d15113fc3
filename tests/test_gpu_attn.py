"""GPU parity of attention over the cache against the fp64 oracle, per workload.

Small cases are compared element by element with the oracle; full-size cases (the
shapes the bench times, same launch configuration) are compared on sampled output
rows that the oracle computes one by one, and on properties that hold at any size.
"""
import numpy as np
import pytest
import torch

from diffusion_serving_gb300 import workloads as wl
from oracle import kvc_oracle as orc
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from diffusion_serving_gb300 import kvc


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def oracle_attend_rows(oracle, b, q_rows, causal=False, q_pos0=0):
    k, v = oracle.keys_values(b)
    return orc.attend(q_rows, k, v, causal=causal, q_pos0=q_pos0)


# ---------------------------------------------------------------------------
# Tiny circular cache, fp32 (7 chunks x 2 rewrites, then reset)
# ---------------------------------------------------------------------------
def run_tiny_ring(w, cache, seed_shift=0):
    oracle = orc.ChronoCache(w.batch, w.kv_heads, w.head_dim, orc.CIRCULAR, sink=w.sink, window=w.window,
                             chunk=w.chunk)
    ww = wl.Workload(**{**w.__dict__, "seed": w.seed + seed_shift})
    outs = []
    for c in range(w.n_chunks):
        cache.advance()
        oracle.advance()
        for r in range(w.rewrites):
            q, k, v = wl.chunk_inputs(ww, c, r, rope_positions=wl.ring_chunk_positions(ww, c))
            cache.write(k.cuda(), v.cuda())
            oracle.write(k.double().numpy(), v.double().numpy())
            out = cache.attend(q.cuda())
            for b in range(w.batch):
                pos = oracle.attended_positions(b)
                slots = torch.tensor([oracle.physical_slot(b, p) for p in pos], device="cuda")
                want = torch.from_numpy(np.stack([oracle.hist_k[b][p] for p in pos])).float()
                assert torch.equal(cache.k_store[b].index_select(0, slots).cpu(), want)
                ref = oracle_attend_rows(oracle, b, q[b].double().numpy())
                assert_close(out[b], ref, f"chunk {c} rewrite {r}")
            outs.append(out.clone())
    return outs


def test_tiny_ring_fp32_with_reset():
    w = wl.TINY_RING
    cache = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.float32, "circular", sink=w.sink,
                        window=w.window, chunk=w.chunk)
    run_tiny_ring(w, cache)
    cache.reset()
    again = run_tiny_ring(w, cache, seed_shift=1)
    fresh = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.float32, "circular", sink=w.sink,
                        window=w.window, chunk=w.chunk)
    new = run_tiny_ring(w, fresh, seed_shift=1)
    for a, b in zip(again, new):
        assert torch.equal(a, b)
    assert cache.get_error() == 0 and fresh.get_error() == 0


# ---------------------------------------------------------------------------
# Active-prefix decode: prefill (causal) then decode steps
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("steps", [wl.DECODE_STEPS])
def test_active_prefix_prefill_and_decode(steps):
    w = wl.DECODE
    T = wl.DECODE_PROMPT
    cache = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.float16, "linear", capacity=w.capacity)
    oracle = orc.ChronoCache(w.batch, w.kv_heads, w.head_dim, orc.LINEAR, capacity=w.capacity)
    q, k, v = wl.chunk_inputs(w, 0, 0, n_q=T, n_kv=T)
    cache.advance(n_tokens=T)
    oracle.advance(n_tokens=T)
    cache.write(k.cuda(), v.cuda())
    oracle.write(k.double().numpy(), v.double().numpy())
    out = cache.attend(q.cuda(), flags=kvc.CAUSAL)
    assert_close(out[0], oracle_attend_rows(oracle, 0, q[0].double().numpy(), causal=True, q_pos0=0), "prefill")
    worst = 0.0
    for i in range(steps):
        q, k, v = wl.chunk_inputs(w, 1 + i, 0, n_q=1, n_kv=1)
        cache.advance(n_tokens=1)
        oracle.advance(n_tokens=1)
        cache.write(k.cuda(), v.cuda())
        oracle.write(k.double().numpy(), v.double().numpy())
        out = cache.attend(q.cuda())
        assert oracle.kv_len[0] == T + i + 1
        e, _ = assert_close(out[0], oracle_attend_rows(oracle, 0, q[0].double().numpy()), f"decode {i}")
        worst = max(worst, e)
    assert cache.row_state()[0][3] == T + steps
    n = T + steps
    want = torch.from_numpy(np.stack([oracle.hist_k[0][p] for p in range(n)])).half()
    assert torch.equal(bits(cache.k_store[0, :n].cpu()), bits(want))
    assert cache.get_error() == 0


@pytest.mark.parametrize("kv_len", [1, 2, 17, 2047, 2048, 2049, 32768])
def test_decode_kernel_lengths(kv_len):
    """Split-KV decode over prefixes that leave empty splits, ragged splits and a full
    32768-slot store, against the oracle and the fp32-FMA kernel."""
    H, Hkv, D, cap = 32, 8, 128, 32768
    cache = kvc.KVCache(1, H, Hkv, D, torch.float16, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(kv_len)
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    cache.set_lengths(kv_len=torch.tensor([kv_len], dtype=torch.int32, device="cuda"))
    q = torch.randn(1, 1, H, D, device="cuda", generator=g).half()
    out = cache.attend(q)
    simt = cache.attend(q, flags=kvc.KERNEL_SIMT)
    ref = orc.attend(to64(q[0]), to64(cache.k_store[0, :kv_len]), to64(cache.v_store[0, :kv_len]))
    assert_close(out[0], ref, "decode")
    assert_close(simt[0], ref, "simt")
    assert cache.get_error() == 0


# ---------------------------------------------------------------------------
# Sink + window streaming (small, complete comparison)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("B,H,Hkv,C,S_c,R_c,n_chunks", [(2, 2, 2, 300, 1, 6, 10), (1, 4, 1, 64, 0, 3, 6),
                                                         (3, 2, 2, 136, 2, 2, 7)])
def test_ring_attention_small(dtype, B, H, Hkv, C, S_c, R_c, n_chunks):
    D = 128
    S, W = S_c * C, (S_c + R_c) * C
    cache = kvc.KVCache(B, H, Hkv, D, dtype, "circular", sink=S, window=W, chunk=C)
    oracle = orc.ChronoCache(B, Hkv, D, orc.CIRCULAR, sink=S, window=W, chunk=C)
    g = torch.Generator().manual_seed(C + n_chunks)
    for c in range(n_chunks):
        cache.advance()
        oracle.advance()
        for r in range(2):
            q = torch.randn(B, C, H, D, generator=g).to(dtype)
            k = torch.randn(B, C, Hkv, D, generator=g).to(dtype)
            v = torch.randn(B, C, Hkv, D, generator=g).to(dtype)
            cache.write(k.cuda(), v.cuda())
            oracle.write(k.double().numpy(), v.double().numpy())
            out = cache.attend(q.cuda())
            for b in range(B):
                assert_close(out[b], oracle_attend_rows(oracle, b, q[b].double().numpy()), f"c{c} r{r} b{b}")
    assert cache.get_error() == 0


# ---------------------------------------------------------------------------
# Sink + window streaming and multi-user batching at full size (sampled rows)
# ---------------------------------------------------------------------------
def sample_rows(gen, n, B, n_q, H):
    b = torch.randint(0, B, (n,), generator=gen)
    i = torch.randint(0, n_q, (n,), generator=gen)
    h = torch.randint(0, H, (n,), generator=gen)
    i[0], i[1] = 0, n_q - 1
    return list(zip(b.tolist(), i.tolist(), h.tolist()))


def check_sampled(out, q, chunks_k, chunks_v, chunk_ids, rows, G, what):
    """Oracle on sampled (b, i, h) rows.  Row b attends the whole chunks chunk_ids[b]
    (chronological order), whose K/V are chunks_k[c][b] and chunks_v[c][b]."""
    for b, i, h in rows:
        ks = torch.cat([chunks_k[c][b, :, h // G] for c in chunk_ids[b]]).double().cpu().numpy()
        vs = torch.cat([chunks_v[c][b, :, h // G] for c in chunk_ids[b]]).double().cpu().numpy()
        ref = orc.attend(to64(q[b, i, h])[None, None, :], ks[:, None, :], vs[:, None, :])[0, 0]
        assert_close(out[b, i, h][None], ref[None], f"{what} (b={b}, i={i}, h={h})")


def full_ring(w, shared_index, rows_per_attend=24, max_chunks=None):
    dtype = wl.DTYPES[w.dtype]
    G = w.heads // w.kv_heads
    cache = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, dtype, "circular", sink=w.sink,
                        window=w.window, chunk=w.chunk)
    oracle = orc.ChronoCache(w.batch, w.kv_heads, w.head_dim, orc.CIRCULAR, sink=w.sink, window=w.window,
                             chunk=w.chunk)
    gen = torch.Generator().manual_seed(w.seed)
    chunks_k, chunks_v = {}, {}
    idx = torch.empty(w.chunk, dtype=torch.int32, device="cuda")
    out = torch.empty(w.batch, w.chunk, w.heads, w.head_dim, dtype=dtype, device="cuda")
    n_chunks = w.n_chunks if max_chunks is None else max_chunks
    for c in range(n_chunks):
        cache.advance()
        oracle.advance()
        pos_c = wl.ring_chunk_positions(w, c)
        if shared_index:
            idx.copy_(torch.tensor([orc.ring_slot(p, w.sink, w.window) for p in pos_c], dtype=torch.int32))
        for r in range(w.rewrites):
            q, k, v = wl.chunk_inputs(w, c, r, device="cuda")
            cache.write(k, v, slots=idx if shared_index else None)
            chunks_k[c], chunks_v[c] = k, v
            cache.attend(q, out)
            # cache contents: the chunk just written sits at its closed-form slots, bit-exact
            slots = [orc.ring_slot(p, w.sink, w.window) for p in pos_c]
            assert slots == list(range(slots[0], slots[0] + w.chunk))
            assert torch.equal(bits(cache.k_store[:, slots[0]:slots[0] + w.chunk]), bits(k))
            assert torch.equal(bits(cache.v_store[:, slots[0]:slots[0] + w.chunk]), bits(v))
            positions = [oracle.attended_positions(b) for b in range(w.batch)]
            chunk_ids = [sorted({p // w.chunk for p in pos}) for pos in positions]
            for b in range(w.batch):
                assert sum(len(range(c * w.chunk, (c + 1) * w.chunk)) for c in chunk_ids[b]) == len(positions[b])
            rows = sample_rows(gen, rows_per_attend, w.batch, w.chunk, w.heads)
            check_sampled(out, q, chunks_k, chunks_v, chunk_ids, rows, G, f"chunk {c} rewrite {r}")
            assert cache.row_state()[0][3] == len(positions[0])
    assert cache.get_error() == 0


@pytest.mark.slow
def test_dit_stream_full_size():
    full_ring(wl.DIT_STREAM, shared_index=False)


@pytest.mark.slow
def test_multi_user_full_size_shared_write_index():
    full_ring(wl.MULTI_USER, shared_index=True, rows_per_attend=16)


# ---------------------------------------------------------------------------
# Ragged cross-attention: packed == padded+kv_len, both == oracle
# ---------------------------------------------------------------------------
def cross_arms(Lq, H, lens, dtype=torch.bfloat16, Lmax=512, device_gen_seed=0):
    D, B = 128, 2
    g = torch.Generator(device="cuda").manual_seed(device_gen_seed + sum(lens))
    q = torch.randn(B, Lq, H, D, device="cuda", generator=g).to(dtype)
    k = torch.randn(B, Lmax, H, D, device="cuda", generator=g).to(dtype)
    v = torch.randn(B, Lmax, H, D, device="cuda", generator=g).to(dtype)
    cu = torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32, device="cuda")
    packed = kvc.KVCache(B, H, H, D, dtype, "packed", capacity=2 * Lmax)
    packed.set_lengths(cu_seqlens=cu)
    packed.write(k, v)
    padded = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=Lmax)
    padded.advance(n_tokens=Lmax)
    padded.write(k, v)
    padded.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    o_packed = packed.attend(q)
    o_kvlen = padded.attend(q)
    unmasked = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=Lmax)
    unmasked.advance(n_tokens=Lmax)
    unmasked.write(k, v)
    o_unmasked = unmasked.attend(q)
    for c in (packed, padded, unmasked):
        assert c.get_error() == 0
    # packed store holds exactly the valid rows, back to back
    for b in range(B):
        lo = int(cu[b])
        assert torch.equal(bits(packed.k_store[lo:lo + lens[b]]), bits(k[b, :lens[b]]))
    return q, k, v, o_packed, o_kvlen, o_unmasked


@pytest.mark.parametrize("lens", [(200, 60), (400, 40), (512, 8), (1, 512), (129, 127)])
def test_cross_attention_small(lens):
    Lq, H = 300, 2
    q, k, v, o_packed, o_kvlen, o_unmasked = cross_arms(Lq, H, lens)
    assert torch.equal(bits(o_packed), bits(o_kvlen))       # same kernel, addressing only
    for b in range(2):
        ref = orc.attend(to64(q[b]), to64(k[b, :lens[b]]), to64(v[b, :lens[b]]))
        assert_close(o_packed[b], ref, f"packed b{b}")
        ref_u = orc.attend(to64(q[b]), to64(k[b]), to64(v[b]))
        assert_close(o_unmasked[b], ref_u, f"unmasked b{b}")


def test_cross_attention_many_items():
    """Ragged cross-attention with 1280 tile pairs (over 8 per SM, so every persistent CTA
    walks many items of both lengths): every row against the oracle."""
    Lq, H, lens = 2 * 128 * 80, 8, (200, 60)
    q, k, v, o_packed, o_kvlen, o_unmasked = cross_arms(Lq, H, lens)
    assert torch.equal(bits(o_packed), bits(o_kvlen))
    for b in range(2):
        ref = orc.attend(to64(q[b]), to64(k[b, :lens[b]]), to64(v[b, :lens[b]]))
        assert_close(o_packed[b], ref, f"packed b{b}")
        ref_u = orc.attend(to64(q[b]), to64(k[b]), to64(v[b]))
        assert_close(o_unmasked[b], ref_u, f"unmasked b{b}")


def test_causal_short_store_many_items():
    """Causal rows of different lengths in a short store (the pair kernel) with 1280 items
    and grouped query heads: the diagonal falls on a different tile and column in each
    row, and the V tail rows zeroed for one item's partial tile are reloaded or re-zeroed
    for the next item that reads that tile."""
    lens = (384, 400, 450, 512, 385, 500, 511, 449)
    B, H, Hkv, D, n_q, cap = len(lens), 80, 8, 128, 384, 512
    cache = kvc.KVCache(B, H, Hkv, D, torch.bfloat16, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(1280)
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    cache.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    q = torch.randn(B, n_q, H, D, device="cuda", generator=g).bfloat16()
    out = cache.attend(q, flags=kvc.CAUSAL)
    for b, n in enumerate(lens):
        ref = orc.attend(to64(q[b]), to64(cache.k_store[b, :n]), to64(cache.v_store[b, :n]), causal=True,
                         q_pos0=n - n_q)
        assert_close(out[b], ref, f"causal row {b} kv_len {n}")
    assert cache.get_error() == 0


@pytest.mark.slow
@pytest.mark.parametrize("skew", list(wl.CROSS_SKEWS))
def test_cross_attention_full_size(skew):
    lens = wl.CROSS_SKEWS[skew]
    H = wl.CROSS.heads
    q, k, v, o_packed, o_kvlen, o_unmasked = cross_arms(wl.CROSS_LQ, H, lens)
    assert torch.equal(bits(o_packed), bits(o_kvlen))
    gen = torch.Generator().manual_seed(len(skew))
    for b, i, h in sample_rows(gen, 24, 2, wl.CROSS_LQ, H):
        ref = orc.attend(to64(q[b, i, h])[None, None], to64(k[b, :lens[b], h])[:, None], to64(v[b, :lens[b], h])[:, None])
        assert_close(o_packed[b, i, h][None], ref[0], f"packed ({b},{i},{h})")
        ref_u = orc.attend(to64(q[b, i, h])[None, None], to64(k[b, :, h])[:, None], to64(v[b, :, h])[:, None])
        assert_close(o_unmasked[b, i, h][None], ref_u[0], f"unmasked ({b},{i},{h})")
    # split-consistency: one branch on its own gives the same bits as the batched run
    for b in range(2):
        one = kvc.KVCache(1, H, H, 128, torch.bfloat16, "packed", capacity=lens[b])
        one.set_lengths(cu_seqlens=torch.tensor([0, lens[b]], dtype=torch.int32, device="cuda"))
        one.write(k[b:b + 1], v[b:b + 1])
        assert torch.equal(bits(one.attend(q[b:b + 1].contiguous())), bits(o_packed[b:b + 1]))


# ---------------------------------------------------------------------------
# Poisoned tail: nothing past kv_len reaches the result
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,big", [(torch.float16, 3e4), (torch.bfloat16, 1e30), (torch.float32, 1e30)])
@pytest.mark.parametrize("kv_len", [1, 130, 300, 511])
def test_poisoned_tail_is_never_read(dtype, big, kv_len):
    B, H, D, cap, n_q = 2, 4, 128, 1024, 150
    cache = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(kv_len)
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    cache.set_lengths(kv_len=torch.tensor([kv_len, kv_len], dtype=torch.int32, device="cuda"))
    q = torch.randn(B, n_q, H, D, device="cuda", generator=g).to(dtype)
    clean = cache.attend(q)
    clean_dec = cache.attend(q[:, :1].contiguous())
    tile_end = min(cap, -(-kv_len // 128) * 128)
    sign = torch.where(torch.rand(B, tile_end - kv_len, H, D, device="cuda", generator=g) > 0.5, 1.0, -1.0)
    cache.k_store[:, kv_len:tile_end] = (sign * big).to(dtype)
    cache.v_store[:, kv_len:tile_end] = (-sign * big).to(dtype)
    cache.k_store[:, tile_end:] = float("nan")
    cache.v_store[:, tile_end:] = float("nan")
    dirty = cache.attend(q)
    dirty_dec = cache.attend(q[:, :1].contiguous())
    assert torch.equal(bits(clean), bits(dirty))
    assert torch.equal(bits(clean_dec), bits(dirty_dec))
    for b in range(B):
        ref = orc.attend(to64(q[b]), to64(cache.k_store[b, :kv_len]), to64(cache.v_store[b, :kv_len]))
        assert_close(dirty[b], ref, "poisoned")
    assert cache.get_error() == 0


# capacity 1024: the query-tile-pair kernel; 2048 and 4096: the one-tile kernel.  The
# longer cases mix whole tiles in range (unmasked path) with the diagonal's masked tiles.
@pytest.mark.parametrize("n_q,kv_len,cap", [(234, 234, 2048), (1, 300, 2048), (130, 300, 2048), (128, 128, 2048),
                                            (300, 1000, 2048), (300, 1000, 1024), (700, 1000, 1024),
                                            (1000, 3000, 4096)])
def test_causal_prefill(n_q, kv_len, cap):
    H, Hkv, D = 8, 2, 128
    cache = kvc.KVCache(1, H, Hkv, D, torch.float16, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(n_q * 7 + kv_len)
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    cache.set_lengths(kv_len=torch.tensor([kv_len], dtype=torch.int32, device="cuda"))
    q = torch.randn(1, n_q, H, D, device="cuda", generator=g).half()
    out = cache.attend(q, flags=kvc.CAUSAL)
    ref = orc.attend(to64(q[0]), to64(cache.k_store[0, :kv_len]), to64(cache.v_store[0, :kv_len]), causal=True,
                     q_pos0=kv_len - n_q)
    assert_close(out[0], ref, "causal")
    assert cache.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("cap,lens", [(1024, (1000, 300, 700)), (4096, (1000, 300, 2900))])
def test_causal_rows_of_different_lengths(dtype, cap, lens):
    """Each row's queries sit at the end of its own active prefix (query i of n_q at
    kv_len_b - n_q + i), so the diagonal falls on a different tile and column in every
    row; bf16 / fp16 run the pair kernel (capacity 1024) or the one-tile kernel (4096),
    fp32 the SIMT kernel."""
    H, Hkv, D, n_q = 8, 2, 128, 300
    cache = kvc.KVCache(len(lens), H, Hkv, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(cap + len(lens))
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    cache.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    q = torch.randn(len(lens), n_q, H, D, device="cuda", generator=g).to(dtype)
    out = cache.attend(q, flags=kvc.CAUSAL)
    for b, n in enumerate(lens):
        ref = orc.attend(to64(q[b]), to64(cache.k_store[b, :n]), to64(cache.v_store[b, :n]), causal=True,
                         q_pos0=n - n_q)
        assert_close(out[b], ref, f"causal row {b} kv_len {n}")
    assert cache.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("cap", [384, 2048])   # short stores: query-tile-pair kernel; long: one-tile kernel
def test_last_tile_chunk_boundaries(dtype, cap):
    """Rows whose last K/V tile ends on and next to every 32-column chunk boundary: the
    tensor-core kernels then read 1, 2, 3 or 4 chunks of that tile's S row and store a
    zero P for the rest.  Slots past kv_len hold NaN; the result must equal the oracle
    and the run with a clean tail, bit for bit."""
    lens = [1, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 128, 129, 161, 255, 256]
    B, H, D, n_q = len(lens), 2, 128, 300
    cache = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(17)
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    cache.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    q = torch.randn(B, n_q, H, D, device="cuda", generator=g).to(dtype)
    clean = cache.attend(q)
    for b, n in enumerate(lens):
        cache.k_store[b, n:] = float("nan")
        cache.v_store[b, n:] = float("nan")
    dirty = cache.attend(q)
    assert torch.equal(bits(clean), bits(dirty))
    for b, n in enumerate(lens):
        ref = orc.attend(to64(q[b]), to64(cache.k_store[b, :n]), to64(cache.v_store[b, :n]))
        assert_close(dirty[b], ref, f"kv_len {n}")
    assert cache.get_error() == 0
