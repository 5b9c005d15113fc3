"""GPU tests of the bounded-wait failure path, without any fault or hang.

Every mbarrier wait in the tensor-core and decode attention kernels gives up after a
limit; the kernel then stops issuing work, lets its own copies and tensor-core
operations finish, frees its tensor memory, sets KVC_DEV_TIMEOUT and returns.  The
testing hook kvc_debug_stall_waits makes the steady-state waits wait, for 200 us, on a
barrier that nothing signals, so that they run out; the test checks that the call returns,
that the error is reported once, and that the next attend on the same handle, with the
default limit, matches the oracle and a fresh handle bit for bit.
"""
import pytest
import torch

from oracle import kvc_oracle as orc
from tests.helpers import assert_close, to64

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from diffusion_serving_gb300 import kvc

CASES = {
    # kernel: (dtype, H, Hkv, capacity, kv_len per row, n_q)
    "pair": (torch.bfloat16, 4, 4, 1024, (1000, 700), 512),      # stores of <= 1024 slots
    "one_tile": (torch.bfloat16, 4, 2, 4096, (4000, 3000), 256),  # longer stores
    "decode": (torch.float16, 32, 8, 32768, (20000, 9000), 1),    # split-KV decode
}


def make(kind, seed):
    dtype, H, Hkv, cap, lens, n_q = CASES[kind]
    c = kvc.KVCache(2, H, Hkv, 128, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(seed)
    c.k_store.normal_(generator=g)
    c.v_store.normal_(generator=g)
    c.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    q = torch.randn(2, n_q, H, 128, device="cuda", generator=g).to(dtype)
    return c, q, lens


@pytest.mark.parametrize("kind", sorted(CASES))
def test_wait_that_runs_out_returns_and_reports(kind):
    c, q, lens = make(kind, 21)
    flags = kvc.DETERMINISTIC
    kvc.kvc_debug_stall_waits(c.handle, 200_000)
    c.attend(q, flags=flags)                           # returns; its output is not defined
    bits = c.get_error()
    assert bits & kvc.DEV_TIMEOUT, f"no wait ran out (error bits {bits:#x})"
    assert c.get_error() == 0                          # reported once, then cleared
    kvc.kvc_debug_stall_waits(c.handle, 0)
    out = c.attend(q, flags=flags)
    assert c.get_error() == 0
    fresh, _, _ = make(kind, 21)
    assert torch.equal(out, fresh.attend(q, flags=flags))
    for b in range(2):
        n = lens[b]
        ref = orc.attend(to64(q[b]), to64(c.k_store[b, :n]), to64(c.v_store[b, :n]))
        assert_close(out[b], ref, f"{kind} row {b} after the timeout")


def test_later_attends_after_a_timeout_run_normally_once_cleared():
    """A timeout left in the error word makes later launches of the chunk kernels return
    at once (they see it before doing any work); once kvc_get_error has cleared it, the
    handle works again."""
    c, q, lens = make("one_tile", 22)
    kvc.kvc_debug_stall_waits(c.handle, 200_000)
    c.attend(q)
    kvc.kvc_debug_stall_waits(c.handle, 0)
    sentinel = torch.full_like(q, 7.0)
    c.attend(q, out=sentinel)                          # the word still holds the timeout
    torch.cuda.synchronize()
    assert torch.all(sentinel == 7.0)
    assert c.get_error() & kvc.DEV_TIMEOUT
    out = c.attend(q)
    assert c.get_error() == 0
    ref = orc.attend(to64(q[0]), to64(c.k_store[0, :lens[0]]), to64(c.v_store[0, :lens[0]]))
    assert_close(out[0], ref, "after clearing")
