"""Seeded synthetic inputs and the workload shapes the pages describe.

This module holds no attention or cache arithmetic: it only draws N(0, 1) tensors
from seeded generators and names the five workload shapes.  Both the CUDA path's
tests/bench and the CPU oracle take their inputs from here, so both see the same
bits.  Nothing here depends on the compiled library.

Keys fed to the tiny circular workload are rotated (RoPE, theta = 1e4, interleaved
pairs, absolute positions) before they reach the cache, as the flashdreams issue
"add an opt-in circular KV policy for streaming attention" requires of keys stored in
a circular cache ("proposed boundary"): the rotation belongs to the model that
produces the keys, so here it is part of synthesising the input.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    layout: str            # "linear" | "circular" | "packed"
    batch: int
    heads: int
    kv_heads: int
    head_dim: int
    chunk: int = 0         # tokens per chunk (circular) / per write
    sink: int = 0
    window: int = 0        # total ring slots, sink included
    capacity: int = 0      # linear: slots per row; packed: total packed slots
    n_chunks: int = 0
    rewrites: int = 1      # denoising writes per chunk (same slots each time)
    seed: int = 0


# Tiny circular cache: 7 chunks x 2 rewrites, then reset (fp32, RoPE'd keys).
TINY_RING = Workload("tiny_ring_fp32_b1h2d64", "f32", "circular", 1, 2, 2, 64,
                     chunk=4, sink=4, window=16, n_chunks=7, rewrites=2, seed=1001)
# Active-prefix decode over a 32768-slot store: prefill 234 then 512 decode steps.
DECODE = Workload("active_prefix_decode_fp16_h32kv8d128", "f16", "linear", 1, 32, 8, 128,
                  capacity=32768, seed=1002)
DECODE_PROMPT, DECODE_STEPS = 234, 512
# Streaming DiT self-attention, cond/uncond rows, sink 3 frames, window 21 frames.
FRAME = 1560
DIT_STREAM = Workload("sink_window_dit_bf16_b2h12d128", "bf16", "circular", 2, 12, 12, 128,
                      chunk=3 * FRAME, sink=3 * FRAME, window=21 * FRAME, n_chunks=10,
                      rewrites=4, seed=1003)
# Homogeneous multi-user batching: 8 users on one chunk timeline, one write index.
MULTI_USER = Workload("multi_user_ring_bf16_b8h40d128", "bf16", "circular", 8, 40, 40, 128,
                      chunk=3 * FRAME, sink=3 * FRAME, window=21 * FRAME, n_chunks=8,
                      rewrites=1, seed=1004)
# Ragged cross-attention: 2 CFG branches, padded Q of 75600 rows, text K/V <= 512.
CROSS_LQ, CROSS_LKV_MAX = 75600, 512
CROSS = Workload("ragged_cross_attn_bf16_b2h40d128", "bf16", "packed", 2, 40, 40, 128,
                 capacity=2 * CROSS_LKV_MAX, seed=1005)
CROSS_SKEWS = {"typical": (200, 60), "moderate": (400, 40), "worst": (512, 8)}

ALL = [TINY_RING, DECODE, DIT_STREAM, MULTI_USER, CROSS]


def step_seed(base: int, chunk: int, rewrite: int, what: int) -> int:
    """Seed of one generated tensor: per workload, chunk, rewrite and tensor kind."""
    return base * 10_000 + chunk * 10 + rewrite + what * 1_000_003


def randn(shape, dtype: str, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) in fp32 from a seeded torch generator, rounded to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    return x.to(DTYPES[dtype])


def rope_rotate(x: torch.Tensor, positions, theta: float = 1e4) -> torch.Tensor:
    """Rotate interleaved pairs of ``x[..., n, H, D]`` by ``pos * theta^(-2i/D)``.

    Computed in fp64 on the CPU, then rounded back to ``x``'s dtype.  ``positions``
    gives the absolute position of each token along dim -3.
    """
    xd = x.to(torch.float64)
    D = x.shape[-1]
    pos = torch.as_tensor(np.asarray(positions, dtype=np.float64))
    inv = theta ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)      # [D/2]
    ang = pos[:, None] * inv[None, :]                                      # [n, D/2]
    c = torch.cos(ang)[:, None, :]
    s = torch.sin(ang)[:, None, :]
    x0, x1 = xd[..., 0::2], xd[..., 1::2]
    out = torch.empty_like(xd)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out.to(x.dtype)


def rope_table(n_positions: int, head_dim: int, theta: float = 1e4) -> torch.Tensor:
    """(cos, sin) of pos * theta^(-2j/D) for every position and pair j, fp64 rounded to
    fp32: shape [n_positions, D/2, 2].  The table a model precomputes once."""
    pos = torch.arange(n_positions, dtype=torch.float64)[:, None]
    inv = theta ** (-torch.arange(0, head_dim, 2, dtype=torch.float64) / head_dim)[None, :]
    ang = pos * inv
    return torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).to(torch.float32).contiguous()


def chunk_inputs(w: Workload, chunk: int, rewrite: int, n_q: int | None = None,
                 n_kv: int | None = None, device="cpu", rope_positions=None):
    """(q, k, v) for one write+attend of workload ``w``.

    q is ``[B, n_q, H, D]``; k and v are ``[B, n_kv, Hkv, D]``.  With
    ``rope_positions`` (absolute token positions of this chunk) q and k are rotated.
    """
    n_kv = w.chunk if n_kv is None else n_kv
    n_q = n_kv if n_q is None else n_q
    q = randn((w.batch, n_q, w.heads, w.head_dim), w.dtype, step_seed(w.seed, chunk, rewrite, 0), device)
    k = randn((w.batch, n_kv, w.kv_heads, w.head_dim), w.dtype, step_seed(w.seed, chunk, rewrite, 1), device)
    v = randn((w.batch, n_kv, w.kv_heads, w.head_dim), w.dtype, step_seed(w.seed, chunk, rewrite, 2), device)
    if rope_positions is not None:
        q = rope_rotate(q.cpu(), rope_positions).to(device)
        k = rope_rotate(k.cpu(), rope_positions).to(device)
    return q, k, v


def ring_chunk_positions(w: Workload, chunk: int):
    return list(range(chunk * w.chunk, (chunk + 1) * w.chunk))


def attention_flops(n_q: int, n_k: int, heads: int, head_dim: int) -> float:
    """Algorithmic flops of unmasked attention, 2 matmuls of 2*n_q*n_k*D per head.

    A count of work, used to turn a measured time into TFLOP/s.
    """
    return 4.0 * n_q * n_k * heads * head_dim


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def l2_flush_bytes() -> int:
    return 256 * 1024 * 1024


def seqlens_to_cu(lengths) -> list[int]:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return cu

