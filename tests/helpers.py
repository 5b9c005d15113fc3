"""Comparison helpers shared by the GPU parity tests (no method arithmetic)."""
from __future__ import annotations

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
