"""The allocation-free decode entry point gives the same output as kvc_attend.

kvc_attend_decode_noalloc serves callers that cannot allocate device memory (code
inside another framework's memory pool, plugins whose host owns every allocation,
steps that must not allocate after graph capture): it keeps the decode kernel's
scratch in an array compiled into the library instead of a caller workspace.  This
file is collected last so that a failure here leaves every other test already run.
"""
import ctypes

import pytest
import torch

from oracle import kvc_oracle as orc
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from diffusion_serving_gb300 import kvc


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_noalloc_decode_matches_kvc_attend_twice(dtype):
    B, H, Hkv, D, cap = 2, 32, 8, 128, 4096
    cache = kvc.KVCache(B, H, Hkv, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(11)
    cache.k_store.normal_(generator=g)
    cache.v_store.normal_(generator=g)
    for call, lens in enumerate(((490, 3000), (4096, 17))):
        cache.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
        q = torch.randn(B, 1, H, D, device="cuda", generator=g).to(dtype)
        want = cache.attend(q)
        got = torch.full_like(q, float("nan"))
        kvc.kvc_attend_decode_noalloc(cache.cfg, cache.k_store, cache.v_store, cache.meta, q, got)
        torch.cuda.synchronize()
        # same tolerance as the other bf16/fp16 comparisons, against kvc_attend and the oracle
        assert_close(got, to64(want), f"call {call} vs kvc_attend")
        for b in range(B):
            ref = orc.attend(to64(q[b]), to64(cache.k_store[b, :lens[b]]), to64(cache.v_store[b, :lens[b]]))
            assert_close(got[b], ref, f"call {call} row {b} vs oracle")
    assert cache.get_error() == 0
    # a third call of another shape (one row, 4 kv heads, a packed store split over more
    # blocks) on the same stream: its counters sit where the calls above left partial
    # data, which the entry point must clear
    lens = (2500,)
    other = kvc.KVCache(1, 16, 4, D, dtype, "packed", capacity=2600)
    other.set_lengths(cu_seqlens=torch.tensor([0, lens[0]], dtype=torch.int32, device="cuda"))
    other.k_store.normal_(generator=g)
    other.v_store.normal_(generator=g)
    q = torch.randn(1, 1, 16, D, device="cuda", generator=g).to(dtype)
    want = other.attend(q)
    got = torch.full_like(q, float("nan"))
    kvc.kvc_attend_decode_noalloc(other.cfg, other.k_store, other.v_store, other.meta, q, got)
    torch.cuda.synchronize()
    assert_close(got, to64(want), "packed call vs kvc_attend")
    ref = orc.attend(to64(q[0]), to64(other.k_store[:lens[0]]), to64(other.v_store[:lens[0]]))
    assert_close(got[0], ref, "packed call vs oracle")
    assert other.get_error() == 0


def test_noalloc_rejects_scratch_beyond_its_array():
    """The library itself refuses (the C call, without the binding's size checks): no
    pointer is touched, so small dummy buffers are enough."""
    cfg = kvc.make_config(1024, 8, 8, 128, torch.float16, "linear", capacity=64)
    t = torch.zeros(16, dtype=torch.float16, device="cuda")
    p = t.data_ptr()
    rc = kvc._lib.kvc_attend_decode_noalloc(ctypes.byref(cfg), p, p, p, p, p, torch.cuda.current_stream().cuda_stream)
    assert rc == kvc.ERR_RANGE
