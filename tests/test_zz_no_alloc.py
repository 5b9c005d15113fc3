"""The allocation-free decode entry point gives the same output as kvc_attend.

kvc_attend_decode_noalloc serves callers that cannot allocate device memory (code
inside another framework's memory pool, plugins whose host owns every allocation,
steps that must not allocate after graph capture): it keeps the decode kernel's
scratch in an array compiled into the library instead of a caller workspace.  This
file is collected last so that a failure here leaves every other test already run.
"""
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


def test_noalloc_rejects_scratch_beyond_its_array():
    cfg = kvc.make_config(1024, 8, 8, 128, torch.float16, "linear", capacity=64)
    t = torch.zeros(16, dtype=torch.float16, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.kvc_attend_decode_noalloc(cfg, t, t, t, t, t)
    assert e.value.code == kvc.ERR_RANGE
