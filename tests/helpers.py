"""Comparison helpers shared by the GPU parity tests: tolerances and error bounds, no
method arithmetic beyond what a bound needs."""
from __future__ import annotations

import math

import numpy as np
import torch

# Output tolerances against the fp64 oracle.
#  fp32: the fish-speech PR's fp32 comparison (rtol 1e-5, atol 1e-6).
#  bf16 / fp16: max-abs 1e-2 and mean-abs 1e-3, with identical row argmax.
TOL = {torch.float32: dict(rtol=1e-5, atol=1e-6),
       torch.float16: dict(max_abs=1e-2, mean_abs=1e-3),
       torch.bfloat16: dict(max_abs=1e-2, mean_abs=1e-3)}
MANTISSA = {torch.float32: 23, torch.float16: 10, torch.bfloat16: 7}


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def ulp(x: np.ndarray, dtype) -> np.ndarray:
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - MANTISSA[dtype])


def argmax_check(got: np.ndarray, ref: np.ndarray, dtype):
    """Row argmax over the last axis must match wherever the oracle's top-1/top-2 gap
    exceeds 2 ulp of the output dtype; inside that gap any index whose oracle value is
    within the gap of the top is accepted.  Returns (mismatches, near-tie rows)."""
    ref2 = ref.reshape(-1, ref.shape[-1])
    got2 = got.reshape(-1, got.shape[-1])
    srt = np.sort(ref2, axis=1)
    top1, top2 = srt[:, -1], srt[:, -2]
    tol = 2 * ulp(top1, dtype)
    decided = (top1 - top2) > tol
    ga = np.argmax(got2, axis=1)
    ra = np.argmax(ref2, axis=1)
    bad_decided = np.sum(decided & (ga != ra))
    picked = ref2[np.arange(len(ga)), ga]
    bad_tied = np.sum(~decided & (picked < top1 - tol))
    return int(bad_decided + bad_tied), int(np.sum(~decided))


def assert_close(got_t: torch.Tensor, ref: np.ndarray, what: str = ""):
    """Compare a GPU output with the fp64 oracle at the tolerance of got_t's dtype."""
    dtype = got_t.dtype
    got = to64(got_t)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    tol = TOL[dtype]
    if dtype == torch.float32:
        bound = tol["atol"] + tol["rtol"] * np.abs(ref)
        worst = np.max(err - bound)
        assert worst <= 0, f"{what}: fp32 max err {err.max():.3e} exceeds rtol/atol"
    else:
        assert err.max() <= tol["max_abs"], f"{what}: max-abs {err.max():.3e}"
        assert err.mean() <= tol["mean_abs"], f"{what}: mean-abs {err.mean():.3e}"
    bad, ties = argmax_check(got, ref, dtype)
    assert bad == 0, f"{what}: {bad} row argmax mismatches ({ties} near-tie rows)"
    return float(err.max()), float(err.mean())


# Error bound of a log-sum-exp computed by the attention kernels (natural log units).
# Each kernel forms scores with fp32 accumulation, exponentiates s * scale * log2(e) - m
# with an approximate exp2, sums the terms in fp32 with a running-max rescale, and
# returns (m + log2 l) * ln 2.  Bounding each step, for a row with fp64 scores s_j,
# softmax weights w_j and n keys:
#  * dot products: each of the D additions of an fp32 accumulation (any order, rounded
#    or truncated) errs by at most one fp32 ulp (2^-23) of a partial sum no larger than
#    sum_d |q_d k_jd|; allowing 2D such steps covers blocked accumulation, so score j
#    errs by B_j = scale * 2D * 2^-23 * sum_d |q_d k_jd|.  The LSE moves by at most the
#    w-weighted mean of the score errors (mean-value theorem; the factor e^(2 max B)
#    covers the weights moving with the scores).
#  * exponent arguments: rounding s * (scale log2 e) and the subtraction of the
#    running max, 2^-23 |s_j| + ln2 2^-24 |t_j| (t_j the argument of exp2), weighted by w.
#  * exponentials: relative error eps_e = 2^-21 per term and per rescale factor (above
#    the relative error PTX states for ex2.approx.f32 and CUDA states for exp2f), with at
#    most T = ceil(n/16) + 160 rescales of the running sum (one per 16-slot tile, plus
#    split and warp merges).
#  * fp32 sums: every term passes through at most A = ceil(n/4) + 64 additions (the
#    longest per-thread chain, the decode kernel's), 2^-24 each.
#  * the final log2, add and multiply by ln 2: 2^-21 (|LSE| + 1).
# A relative error x of the sum moves the log by at most x / (1 - x).
EPS_EXP2 = 2.0 ** -21


def lse_error_bound(q, k, scale, lse_ref):
    """Per-row bound [n_q, H] on |LSE_gpu - LSE_exact| for fp64 q [n_q, H, D], the keys
    k [n, Hkv, D] one row attends and the oracle's LSE [n_q, H] (rows with keys)."""
    n_q, H, D = q.shape
    n, Hkv, _ = k.shape
    G = H // Hkv
    T = -(-n // 16) + 160
    A = -(-n // 4) + 64
    rel_sum = (2 + T) * EPS_EXP2 + A * 2.0 ** -24
    out = np.empty((n_q, H))
    for h in range(H):
        kh = k[:, h // G, :]
        s = scale * (q[:, h, :] @ kh.T)                          # [n_q, n]
        w = np.exp(s - lse_ref[:, h][:, None])
        B = scale * 2 * D * 2.0 ** -23 * (np.abs(q[:, h, :]) @ np.abs(kh).T)
        t = (s - s.max(axis=1, keepdims=True)) / math.log(2)
        dots = np.exp(2 * B.max(axis=1)) * (w * B).sum(axis=1)
        args = (w * (2.0 ** -23 * np.abs(s) + math.log(2) * 2.0 ** -24 * np.abs(t))).sum(axis=1)
        out[:, h] = dots + args + rel_sum / (1 - rel_sum) + 2.0 ** -21 * (np.abs(lse_ref[:, h]) + 1)
    return out


def merge_lse_error_bound(lse_a, lse_b, bound_a, bound_b):
    """Bound on the merged LSE: the merge is 1-Lipschitz in its two inputs (max of their
    bounds), plus its own fp32 arithmetic (expf within 2 ulp, logf within 1 ulp, the
    rounding of the difference of the inputs and of the final add)."""
    L = np.logaddexp(lse_a, lse_b)
    own = 2.0 ** -20 + 2.0 ** -23 * (np.abs(L) + np.abs(lse_a - lse_b))
    return np.maximum(bound_a, bound_b) + own
