"""GPU tests of the write with RoPE fused into the K half (kvc_write_rope).

Keys are rotated at their absolute positions before storage (flashdreams issue "add an
opt-in circular KV policy for streaming attention", "proposed boundary").  The GPU turns
each pair in fp32 and rounds once to the store type; the oracle turns it in fp64 from the
same (cos, sin) table.  The stored K therefore matches the oracle rounded to the store
type except where the exact value lies within fp32 rounding of a rounding boundary: every
element within 1 ulp of the store type, and nearly all equal.  V is copied bit-exact.
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

MANT = {torch.float32: 23, torch.float16: 10, torch.bfloat16: 7}


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def check_rotated(got, x, positions, table, dtype):
    """got: stored K rows [n, Hkv, D] (dtype); x: raw rows; returns the fraction exact."""
    ref = orc.rope_apply(to64(x), positions, table)
    want = torch.from_numpy(ref).to(dtype)
    g64, w64 = to64(got.cpu()), to64(want)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(w64), 1e-30))) - MANT[dtype])
    # fp32 arithmetic on the pair: a few fp32 roundings of the operands' magnitude
    xx = np.abs(to64(x))
    pair = np.repeat(xx[..., 0::2] + xx[..., 1::2], 2, axis=-1)
    tol = np.maximum(ulp * 1.0001, 4 * 2.0 ** -24 * pair)
    assert np.all(np.abs(g64 - w64) <= tol), "rotated K off by more than 1 ulp of the store type"
    return float(np.mean(bits(got.cpu()).numpy() == bits(want).numpy()))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_ring_write_rope_positions_and_attention(dtype):
    B, H, Hkv, D, C, S, W = 2, 4, 2, 128, 24, 24, 96
    table = wl.rope_table(4096, D)
    tab_np = table.numpy()
    d_table = table.cuda()
    cache = kvc.KVCache(B, H, Hkv, D, dtype, "circular", sink=S, window=W, chunk=C)
    oracle = orc.ChronoCache(B, Hkv, D, orc.CIRCULAR, sink=S, window=W, chunk=C)
    g = torch.Generator().manual_seed(3)
    exact = []
    for c in range(9):                          # fill, two wraps, rewrites
        cache.advance()
        oracle.advance()
        for rw in range(2):
            k = torch.randn(B, C, Hkv, D, generator=g).to(dtype)
            v = torch.randn(B, C, Hkv, D, generator=g).to(dtype)
            q = torch.randn(B, C, H, D, generator=g).to(dtype)
            cache.write_rope(k.cuda(), v.cuda(), d_table)
            pos = list(range(c * C, (c + 1) * C))
            slot0 = orc.ring_slot(c * C, S, W)
            for b in range(B):
                exact.append(check_rotated(cache.k_store[b, slot0:slot0 + C], k[b], pos, tab_np, dtype))
                assert torch.equal(bits(cache.v_store[b, slot0:slot0 + C].cpu()), bits(v[b]))
            # the oracle history keeps the GPU's stored (rotated) K rows, so attention is
            # compared on identical inputs
            stored = cache.k_store[:, slot0:slot0 + C].cpu()
            oracle.write(to64(stored), to64(v))
            out = cache.attend(q.cuda())
            for b in range(B):
                kk, vv = oracle.keys_values(b)
                assert_close(out[b], orc.attend(to64(q[b]), kk, vv), f"chunk {c}")
    assert np.mean(exact) > 0.99
    assert cache.get_error() == 0


def test_linear_write_rope_uses_slots_as_positions():
    B, Hkv, D, cap = 2, 4, 64, 512
    table = wl.rope_table(cap, D)
    cache = kvc.KVCache(B, Hkv, Hkv, D, torch.bfloat16, "linear", capacity=cap)
    k = torch.randn(B, 7, Hkv, D).bfloat16()
    slots = [5, 100, 101, 300, 0, 511, 256]
    cache.write_rope(k.cuda(), k.cuda(), table.cuda(), slots=torch.tensor(slots, dtype=torch.int32, device="cuda"))
    for b in range(B):
        got = cache.k_store[b, slots]
        assert check_rotated(got, k[b], slots, table.numpy(), torch.bfloat16) > 0.98
    assert cache.get_error() == 0


def test_packed_write_rope_positions_start_at_zero_per_row():
    lens = (13, 5)
    Hkv, D = 2, 128
    table = wl.rope_table(64, D)
    cache = kvc.KVCache(2, Hkv, Hkv, D, torch.float16, "packed", capacity=32)
    cache.set_lengths(cu_seqlens=torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32, device="cuda"))
    k = torch.randn(2, 16, Hkv, D).half()
    cache.write_rope(k.cuda(), k.cuda(), table.cuda())
    lo = 0
    for b in range(2):
        got = cache.k_store[lo:lo + lens[b]]
        assert check_rotated(got, k[b, :lens[b]], list(range(lens[b])), table.numpy(), torch.float16) > 0.98
        lo += lens[b]
    assert cache.get_error() == 0


def test_positions_past_the_table_are_reported_and_skipped():
    C, D = 8, 64
    cache = kvc.KVCache(1, 2, 2, D, torch.bfloat16, "circular", sink=C, window=4 * C, chunk=C)
    table = wl.rope_table(2 * C, D).cuda()             # covers chunks 0 and 1 only
    cache.k_store.zero_()
    k = torch.randn(1, C, 2, D, device="cuda").bfloat16()
    for c in range(3):
        cache.advance()
        cache.write_rope(k, k, table)
        err = cache.get_error()
        assert err == (kvc.DEV_BAD_POS if c == 2 else 0)
    assert torch.all(cache.k_store[0, 2 * C:3 * C] == 0)
