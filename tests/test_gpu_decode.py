"""GPU parity of the split-KV decode kernel (one query token per row) across its shapes.

The decode step of the fish-speech PR "perf(text2semantic): pass only active KV cache
prefix to SDPA" ("Change": step i attends kv_len = T + i + 1 slots; GQA heads share one
read of their kv head).  Every instantiation (fp16 / bf16, D = 64 / 128, G = 1, 2, 4, 8)
is compared with the oracle on rows whose lengths fall on and around the kernel's
112-slot tiles and 16-slot warp slices, on packed rows (the TensorRT-LLM PR "FA4
variable-length cross-attention", Description), and over repeated calls, which reuse
the workspace's ticket and tile-claim counters.
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

# lengths: a single slot, a warp slice, a ragged warp slice, one tile, one past a tile,
# the last length one block streams alone and the first one split over blocks (4 tiles
# and one slot more), one past 5 tiles, several tiles with a ragged tail
LENS = (1, 16, 17, 112, 113, 448, 449, 561, 1000, 2900)


def linear_cache(dtype, H, Hkv, D, lens, cap, seed):
    c = kvc.KVCache(len(lens), H, Hkv, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(seed)
    c.k_store.normal_(generator=g)
    c.v_store.normal_(generator=g)
    c.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    return c, g


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_every_instantiation(dtype, D, G):
    Hkv = 2
    H = G * Hkv
    c, g = linear_cache(dtype, H, Hkv, D, LENS, 3000, 100 * G + D)
    q = torch.randn(len(LENS), 1, H, D, device="cuda", generator=g).to(dtype)
    out = c.attend(q)
    for b, n in enumerate(LENS):
        ref = orc.attend(to64(q[b]), to64(c.k_store[b, :n]), to64(c.v_store[b, :n]))
        assert_close(out[b], ref, f"row {b} kv_len {n}")
    assert c.get_error() == 0


def test_decode_packed_rows():
    lens = (5, 300, 129, 1)
    H, Hkv, D = 16, 4, 128
    cap = sum(lens)
    c = kvc.KVCache(len(lens), H, Hkv, D, torch.bfloat16, "packed", capacity=cap)
    c.set_lengths(cu_seqlens=torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32, device="cuda"))
    g = torch.Generator(device="cuda").manual_seed(7)
    c.k_store.normal_(generator=g)
    c.v_store.normal_(generator=g)
    q = torch.randn(len(lens), 1, H, D, device="cuda", generator=g).bfloat16()
    out = c.attend(q)
    lo = 0
    for b, n in enumerate(lens):
        ref = orc.attend(to64(q[b]), to64(c.k_store[lo:lo + n]), to64(c.v_store[lo:lo + n]))
        assert_close(out[b], ref, f"packed row {b}")
        lo += n
    assert c.get_error() == 0


def test_decode_repeated_calls_and_changing_lengths():
    """Calls back to back, with lengths that change between them: each call must start
    from zeroed counters (the last block of each (row, kv head) resets them)."""
    H, Hkv, D = 32, 8, 128
    c, g = linear_cache(torch.float16, H, Hkv, D, [4000, 7], 8192, 11)
    q = torch.randn(2, 1, H, D, device="cuda", generator=g).half()
    for lens in ([4000, 7], [8192, 1], [3, 5000], [4000, 7]):
        c.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
        first = c.attend(q)                          # 8192 slots: tiles past the fixed ones are claimed
        fixed = c.attend(q, flags=kvc.DETERMINISTIC)
        again = c.attend(q, flags=kvc.DETERMINISTIC)
        assert torch.equal(fixed, again)
        for b, n in enumerate(lens):
            ref = orc.attend(to64(q[b]), to64(c.k_store[b, :n]), to64(c.v_store[b, :n]))
            assert_close(first[b], ref, f"lens {lens} row {b}")
            assert_close(fixed[b], ref, f"lens {lens} row {b} fixed tiles")
    assert c.get_error() == 0


def test_decode_poisoned_tail_is_not_read():
    """Slots past kv_len hold NaN and huge values; the output must not change."""
    H, Hkv, D, n = 8, 2, 128, 150          # 150 = one full tile + a ragged warp slice
    c, g = linear_cache(torch.bfloat16, H, Hkv, D, [n], 1024, 5)
    q = torch.randn(1, 1, H, D, device="cuda", generator=g).bfloat16()
    clean = c.attend(q)
    c.k_store[0, n:n + 80] = 1e30
    c.v_store[0, n:n + 80] = -1e30
    c.k_store[0, n + 80:] = float("nan")
    c.v_store[0, n + 80:] = float("nan")
    poisoned = c.attend(q)
    assert torch.equal(clean, poisoned)
    assert c.get_error() == 0


def test_decode_long_row_claimed_and_fixed_tiles():
    """A 32768-slot row has more tiles than the blocks' fixed first tiles: by default
    the rest are claimed at run time (result equal to the oracle, last bits may vary
    between calls); with KVC_DETERMINISTIC every block keeps a fixed set and repeated
    calls agree bit for bit."""
    H, Hkv, D, n = 32, 8, 128, 32768
    c, g = linear_cache(torch.float16, H, Hkv, D, [n], n, 21)
    q = torch.randn(1, 1, H, D, device="cuda", generator=g).half()
    ref = orc.attend(to64(q[0]), to64(c.k_store[0]), to64(c.v_store[0]))
    claimed = c.attend(q)
    fixed = [c.attend(q, flags=kvc.DETERMINISTIC) for _ in range(3)]
    assert_close(claimed[0], ref, "claimed tiles")
    assert_close(fixed[0][0], ref, "fixed tiles")
    assert torch.equal(fixed[0], fixed[1]) and torch.equal(fixed[0], fixed[2])
    assert (claimed.float() - fixed[0].float()).abs().max().item() < 1e-2
    assert c.get_error() == 0
