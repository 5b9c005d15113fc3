"""GPU tests of the write with RoPE fused into the K half (kvc_write_rope).

Keys are rotated at their absolute positions before storage (flashdreams issue "add an
opt-in circular KV policy for streaming attention", "proposed boundary").  The store must
hold exactly what the oracle's ``rope_store`` gives: the exact rotation of the stored
input by the caller's (cos, sin) table, rounded once to nearest-even in the store type.
Every element is compared bit for bit, for bf16, fp16 and fp32 stores, in circular,
linear-with-slots and packed layouts, and on constructed ties and near-ties of the
rounding.  V is copied bit-exact.
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

FMT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def bits(t):
    t = t.contiguous()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def check_rotated(got, x, positions, table, dtype):
    """got: stored K rows [n, Hkv, D] (dtype); x: the rows written.  Bit-exact."""
    want = torch.from_numpy(orc.rope_store(to64(x), positions, table, FMT[dtype])).to(dtype)
    g, w = bits(got.cpu()), bits(want)
    bad = int((g != w).sum())
    assert bad == 0, f"{bad} of {g.numel()} rotated K elements differ from the once-rounded rotation"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_ring_write_rope_positions_and_attention(dtype):
    B, H, Hkv, D, C, S, W = 2, 4, 2, 128, 24, 24, 96
    table = wl.rope_table(4096, D)
    tab_np = table.numpy()
    d_table = table.cuda()
    cache = kvc.KVCache(B, H, Hkv, D, dtype, "circular", sink=S, window=W, chunk=C)
    oracle = orc.ChronoCache(B, Hkv, D, orc.CIRCULAR, sink=S, window=W, chunk=C)
    g = torch.Generator().manual_seed(3)
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
                check_rotated(cache.k_store[b, slot0:slot0 + C], k[b], pos, tab_np, dtype)
                assert torch.equal(bits(cache.v_store[b, slot0:slot0 + C].cpu()), bits(v[b]))
            # the oracle history keeps the GPU's stored (rotated) K rows, so attention is
            # compared on identical inputs
            stored = cache.k_store[:, slot0:slot0 + C].cpu()
            oracle.write(to64(stored), to64(v))
            out = cache.attend(q.cuda())
            for b in range(B):
                kk, vv = oracle.keys_values(b)
                assert_close(out[b], orc.attend(to64(q[b]), kk, vv), f"chunk {c}")
    assert cache.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_linear_write_rope_uses_slots_as_positions(dtype):
    B, Hkv, D, cap = 2, 4, 64, 512
    table = wl.rope_table(cap, D)
    cache = kvc.KVCache(B, Hkv, Hkv, D, dtype, "linear", capacity=cap)
    k = torch.randn(B, 7, Hkv, D).to(dtype)
    slots = [5, 100, 101, 300, 0, 511, 256]
    cache.write_rope(k.cuda(), k.cuda(), table.cuda(), slots=torch.tensor(slots, dtype=torch.int32, device="cuda"))
    for b in range(B):
        check_rotated(cache.k_store[b, slots], k[b], slots, table.numpy(), dtype)
    assert cache.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_packed_write_rope_positions_start_at_zero_per_row(dtype):
    lens = (13, 5)
    Hkv, D = 2, 128
    table = wl.rope_table(64, D)
    cache = kvc.KVCache(2, Hkv, Hkv, D, dtype, "packed", capacity=32)
    cache.set_lengths(cu_seqlens=torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32, device="cuda"))
    k = torch.randn(2, 16, Hkv, D).to(dtype)
    cache.write_rope(k.cuda(), k.cuda(), table.cuda())
    lo = 0
    for b in range(2):
        check_rotated(cache.k_store[lo:lo + lens[b]], k[b, :lens[b]], list(range(lens[b])), table.numpy(), dtype)
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


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_write_rope_rounds_ties_and_near_ties_once(dtype):
    """Constructed cases where rounding twice would go wrong: products exactly on a
    rounding midpoint of the store type (ties to even), and pushed off it by a second
    product below half an fp64 ulp (only the exact rest decides), plus many binades,
    subnormal results and overflow.  One table row per token, one pair per case."""
    from tests.test_oracle import rope_cases
    fmt = FMT[dtype]
    D = 64
    n_tok = 96
    x, cs = rope_cases(fmt, n_tok * D // 2, 11)
    k = torch.from_numpy(x.reshape(1, n_tok, 1, D)).to(dtype)
    table = torch.from_numpy(cs.reshape(n_tok, D // 2, 2).astype(np.float32))
    cache = kvc.KVCache(1, 1, 1, D, dtype, "linear", capacity=n_tok)
    slots = torch.arange(n_tok, dtype=torch.int32, device="cuda")
    cache.write_rope(k.cuda(), k.cuda(), table.cuda(), slots=slots)
    check_rotated(cache.k_store[0], k[0], list(range(n_tok)), table.numpy(), dtype)
    assert cache.get_error() == 0
