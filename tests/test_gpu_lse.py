"""GPU tests of attention with log-sum-exp output and of the two-way merge.

The LSE of each row (ln sum_j exp(scale q.k_j)) lets attentions over disjoint key sets
be combined exactly (the forward_with_lse of the TensorRT-LLM PR "FA4 variable-length
cross-attention").  Checked for every kernel against the oracle, and by splitting one
store's keys into two stores and merging.
"""
import numpy as np
import pytest
import torch

from oracle import kvc_oracle as orc
from tests.helpers import assert_close, lse_error_bound, merge_lse_error_bound, to64

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from diffusion_serving_gb300 import kvc



def check_lse(got, q, k, ref_l, what=""):
    """Every row's LSE within the bound derived from the kernels' arithmetic."""
    bound = lse_error_bound(q, k, orc.default_scale(q.shape[-1]), ref_l)
    err = np.abs(got - ref_l)
    assert np.all(err <= bound), f"{what}: LSE error {err.max():.3e} above its bound at {np.argmax(err - bound)}"
    return bound


def filled_linear(B, H, Hkv, D, dtype, cap, lens, seed):
    c = kvc.KVCache(B, H, Hkv, D, dtype, "linear", capacity=cap)
    g = torch.Generator(device="cuda").manual_seed(seed)
    c.k_store.normal_(generator=g)
    c.v_store.normal_(generator=g)
    c.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    return c, g


@pytest.mark.parametrize("dtype,n_q,flags,H,Hkv", [
    (torch.bfloat16, 300, 0, 4, 4),          # tensor-core kernel
    (torch.float16, 1, 0, 8, 2),             # split-KV decode
    (torch.float32, 37, 0, 2, 2),            # fp32-FMA kernel
    (torch.bfloat16, 40, 256, 4, 2),         # fp32-FMA kernel forced on bf16
])
def test_attend_lse_matches_oracle(dtype, n_q, flags, H, Hkv):
    B, D, cap = 2, 128, 3000
    lens = [2049, 130]
    c, g = filled_linear(B, H, Hkv, D, dtype, cap, lens, n_q + H)
    q = torch.randn(B, n_q, H, D, device="cuda", generator=g).to(dtype)
    out, lse = c.attend_lse(q, flags=flags)
    plain = c.attend(q, flags=flags)
    assert torch.equal(out, plain)                      # the LSE costs nothing in the output
    for b in range(B):
        ref_o, ref_l = orc.attend_lse(to64(q[b]), to64(c.k_store[b, :lens[b]]), to64(c.v_store[b, :lens[b]]))
        assert_close(out[b], ref_o, f"row {b}")
        check_lse(lse[b].cpu().double().numpy(), to64(q[b]), to64(c.k_store[b, :lens[b]]), ref_l, f"row {b}")
    assert c.get_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_split_then_merge_equals_whole(dtype):
    """Keys split across two stores, attended separately, merged: equal to one store."""
    B, H, D, n_q = 1, 4, 128, 200
    n_a, n_b = 700, 333
    g = torch.Generator(device="cuda").manual_seed(9)
    k = torch.randn(B, n_a + n_b, H, D, device="cuda", generator=g).to(dtype)
    v = torch.randn(B, n_a + n_b, H, D, device="cuda", generator=g).to(dtype)
    q = torch.randn(B, n_q, H, D, device="cuda", generator=g).to(dtype)
    whole = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=n_a + n_b)
    whole.advance(n_tokens=n_a + n_b)
    whole.write(k, v)
    part_a = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=n_a)
    part_a.advance(n_tokens=n_a)
    part_a.write(k[:, :n_a].contiguous(), v[:, :n_a].contiguous())
    part_b = kvc.KVCache(B, H, H, D, dtype, "linear", capacity=n_b)
    part_b.advance(n_tokens=n_b)
    part_b.write(k[:, n_a:].contiguous(), v[:, n_a:].contiguous())
    o_w, l_w = whole.attend_lse(q)
    o_a, l_a = part_a.attend_lse(q)
    o_b, l_b = part_b.attend_lse(q)
    merged = torch.empty_like(o_a)
    l_m = torch.empty_like(l_a)
    rows = B * n_q * H
    kvc.kvc_merge(dtype, rows, D, o_a, l_a, o_b, l_b, merged, l_m)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.attend_lse(to64(q[0]), to64(k[0]), to64(v[0]))
    _, ref_a = orc.attend_lse(to64(q[0]), to64(k[0, :n_a]), to64(v[0, :n_a]))
    _, ref_b = orc.attend_lse(to64(q[0]), to64(k[0, n_a:]), to64(v[0, n_a:]))
    assert_close(merged[0], ref_o, "merged vs oracle")
    b_a = check_lse(l_a[0].cpu().double().numpy(), to64(q[0]), to64(k[0, :n_a]), ref_a, "half a")
    b_b = check_lse(l_b[0].cpu().double().numpy(), to64(q[0]), to64(k[0, n_a:]), ref_b, "half b")
    b_w = check_lse(l_w[0].cpu().double().numpy(), to64(q[0]), to64(k[0]), ref_l, "whole")
    b_m = merge_lse_error_bound(ref_a, ref_b, b_a, b_b)
    assert np.all(np.abs(l_m[0].cpu().double().numpy() - ref_l) <= b_m), "merged LSE above its bound"
    # the merged result agrees with the one-store attention within rounding of the halves
    assert (merged.float() - o_w.float()).abs().max().item() < 1e-2
    assert np.all(np.abs((l_m - l_w)[0].cpu().double().numpy()) <= b_m + b_w)


def test_merge_rows_without_keys():
    rows, D = 64, 128
    oa = torch.randn(rows, D, device="cuda").bfloat16()
    ob = torch.randn(rows, D, device="cuda").bfloat16()
    la = torch.randn(rows, device="cuda")
    lb = torch.randn(rows, device="cuda")
    la[:8] = float("-inf")                               # half a: no key for rows 0-7
    lb[:4] = float("-inf")                               # rows 0-3: no key at all
    out = torch.empty_like(oa)
    lo = torch.empty_like(la)
    kvc.kvc_merge(torch.bfloat16, rows, D, oa, la, ob, lb, out, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.merge_lse(to64(oa), la.double().cpu().numpy(), to64(ob), lb.double().cpu().numpy())
    assert torch.all(out[:4] == 0) and torch.all(torch.isneginf(lo[:4]))
    assert np.abs(to64(out) - ref_o).max() < 1e-2
    fin = np.isfinite(ref_l)
    la64, lb64 = la.double().cpu().numpy(), lb.double().cpu().numpy()
    zero = np.zeros(rows)
    with np.errstate(invalid="ignore"):
        bound = merge_lse_error_bound(la64, lb64, zero, zero)
    bound = np.where(np.isfinite(la64) & np.isfinite(lb64), bound, 2.0 ** -20 + 2.0 ** -23 * np.abs(ref_l))
    assert np.all(np.abs(lo.double().cpu().numpy()[fin] - ref_l[fin]) <= bound[fin])


@pytest.mark.parametrize("case", ["vector_ragged", "odd_head_dim", "unaligned"])
def test_merge_paths_match_oracle(case):
    """A ragged row count, a row size that is not a multiple of 16 bytes and buffers off
    a 16-byte boundary all give the oracle's merge, and rows without keys give 0 and
    -inf."""
    rows, D = (1001, 128) if case != "odd_head_dim" else (257, 72)
    g = torch.Generator(device="cuda").manual_seed(31)
    pad = 1 if case == "unaligned" else 0
    base_a = torch.randn(rows * D + pad, device="cuda", generator=g).bfloat16()
    base_b = torch.randn(rows * D + pad, device="cuda", generator=g).bfloat16()
    oa, ob = base_a[pad:].view(rows, D), base_b[pad:].view(rows, D)
    la = torch.randn(rows, device="cuda", generator=g) * 4
    lb = torch.randn(rows, device="cuda", generator=g) * 4
    la[5] = float("-inf")
    la[7] = lb[7] = float("-inf")
    out_base = torch.full((rows * D + pad,), float("nan"), device="cuda").bfloat16()
    out = out_base[pad:].view(rows, D)
    lo = torch.empty_like(la)
    kvc.kvc_merge(torch.bfloat16, rows, D, oa, la, ob, lb, out, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.merge_lse(to64(oa), la.double().cpu().numpy(), to64(ob), lb.double().cpu().numpy())
    got = to64(out)
    assert np.all(np.isfinite(got))
    # the fp32 combination (weights from expf / logf / a division: a few ulp each) then
    # one bf16 rounding (unit roundoff 2^-8): |err| <= 2^-8 |o| + 2^-19 (|wa oa| + |wb ob|)
    la64, lb64 = la.double().cpu().numpy(), lb.double().cpu().numpy()
    safe = np.where(np.isfinite(ref_l), ref_l, 0.0)
    wa = np.where(np.isfinite(la64), np.exp(la64 - safe), 0.0)[:, None]
    wb = np.where(np.isfinite(lb64), np.exp(lb64 - safe), 0.0)[:, None]
    mag = np.abs(wa * to64(oa)) + np.abs(wb * to64(ob))
    assert np.all(np.abs(got - ref_o) <= 2.0 ** -8 * np.abs(ref_o) + 2.0 ** -19 * mag)
    assert torch.all(out[7] == 0) and torch.isneginf(lo[7])
    fin = np.isfinite(ref_l)
    assert np.allclose(lo.double().cpu().numpy()[fin], ref_l[fin], rtol=1e-6, atol=1e-5)


UNIT_ROUNDOFF = {torch.float32: 2.0 ** -24, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}
# half the spacing of the type's subnormals: the absolute rounding error below its normal range
SUBNORMAL_HALF_STEP = {torch.float32: 2.0 ** -150, torch.float16: 2.0 ** -25, torch.bfloat16: 2.0 ** -134}


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [128, 72])                 # 16-byte chunk path, scalar path
@pytest.mark.parametrize("alias", ["none", "a", "b"])   # out written over o_a or o_b
def test_merge_dtypes_and_in_place(dtype, D, alias):
    """The merge in every store type, on both kernel paths, into a separate buffer and in
    place over either input: the oracle's merge within one rounding to the type plus the
    fp32 weights' error (or half a subnormal step, for results below the type's normal
    range), rows without keys 0 and -inf."""
    rows = 777
    g = torch.Generator(device="cuda").manual_seed(D + len(alias))
    oa = torch.randn(rows, D, device="cuda", generator=g).to(dtype)
    ob = torch.randn(rows, D, device="cuda", generator=g).to(dtype)
    la = torch.randn(rows, device="cuda", generator=g) * 4
    lb = torch.randn(rows, device="cuda", generator=g) * 4
    la[3] = float("-inf")
    la[9] = lb[9] = float("-inf")
    oa64, ob64 = to64(oa), to64(ob)
    la64, lb64 = la.double().cpu().numpy(), lb.double().cpu().numpy()
    out = {"none": torch.empty_like(oa), "a": oa, "b": ob}[alias]
    lo = torch.empty_like(la)
    kvc.kvc_merge(dtype, rows, D, oa, la, ob, lb, out, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = orc.merge_lse(oa64, la64, ob64, lb64)
    safe = np.where(np.isfinite(ref_l), ref_l, 0.0)
    wa = np.where(np.isfinite(la64), np.exp(la64 - safe), 0.0)[:, None]
    wb = np.where(np.isfinite(lb64), np.exp(lb64 - safe), 0.0)[:, None]
    mag = np.abs(wa * oa64) + np.abs(wb * ob64)
    got = to64(out)
    bound_o = UNIT_ROUNDOFF[dtype] * np.abs(ref_o) + 2.0 ** -19 * mag + SUBNORMAL_HALF_STEP[dtype]
    err = np.abs(got - ref_o)
    assert np.all(err <= bound_o), f"worst {np.unravel_index(np.argmax(err - bound_o), err.shape)}"
    assert torch.all(out[9] == 0) and torch.isneginf(lo[9])
    fin = np.isfinite(ref_l)
    with np.errstate(invalid="ignore"):
        bound = merge_lse_error_bound(la64, lb64, np.zeros(rows), np.zeros(rows))
    bound = np.where(np.isfinite(la64) & np.isfinite(lb64), bound, 2.0 ** -20 + 2.0 ** -23 * np.abs(ref_l))
    assert np.all(np.abs(lo.double().cpu().numpy()[fin] - ref_l[fin]) <= bound[fin])
