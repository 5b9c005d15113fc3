"""GPU tests of shared length layouts (kvc_lengths_*, kvc_use_lengths).

A length layout is prepared once and read by many handles, e.g. every layer of a model
attending the same ragged text K/V (TensorRT-LLM PR "FA4 variable-length
cross-attention", Description: cu_seqlens_kv prepared once and cached, reused across
layers and denoising steps).  Handles that read a shared layout must give exactly what
they give with the same lengths in their own meta block.
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


def packed_layers(n_layers, lens, H, D, dtype, cap, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    layers = []
    for _ in range(n_layers):
        c = kvc.KVCache(len(lens), H, H, D, dtype, "packed", capacity=cap)
        c.k_store.normal_(generator=g)
        c.v_store.normal_(generator=g)
        layers.append(c)
    return layers, g


def test_packed_layers_share_one_layout():
    """Six layers' cross-attention over one prepared cu_seqlens: bit-identical to each
    layer setting its own, and to the oracle; then a second step's layout."""
    H, D, cap, n_q = 8, 128, 1024, 300
    layers, g = packed_layers(6, (200, 60), H, D, torch.bfloat16, cap, 5)
    shared = kvc.KVLengths(2, "packed", cap)
    for lens in ((200, 60), (512, 8)):
        cu = torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32, device="cuda")
        shared.set(cu_seqlens=cu)
        q = torch.randn(2, n_q, H, D, device="cuda", generator=g).bfloat16()
        for i, c in enumerate(layers):
            c.use_lengths(shared)
            got = c.attend(q)
            c.use_lengths(None)
            c.set_lengths(cu_seqlens=cu)
            assert torch.equal(got, c.attend(q)), f"layer {i}"
            if i == 0:
                lo = 0
                for b, n in enumerate(lens):
                    ref = orc.attend(to64(q[b]), to64(c.k_store[lo:lo + n]), to64(c.v_store[lo:lo + n]))
                    assert_close(got[b], ref, f"lens {lens} row {b}")
                    lo += n
            assert c.get_error() == 0


@pytest.mark.parametrize("n_q", [1, 64])
def test_linear_layers_share_kv_len(n_q):
    """Per-row active prefixes shared by layers of a linear store, through the chunk and
    the decode kernels."""
    B, H, Hkv, D, cap = 2, 16, 4, 128, 2048
    g = torch.Generator(device="cuda").manual_seed(7)
    layers = [kvc.KVCache(B, H, Hkv, D, torch.float16, "linear", capacity=cap) for _ in range(3)]
    for c in layers:
        c.k_store.normal_(generator=g)
        c.v_store.normal_(generator=g)
    shared = kvc.KVLengths(B, "linear", cap)
    kv_len = torch.tensor([1500, 77], dtype=torch.int32, device="cuda")
    shared.set(kv_len=kv_len)
    q = torch.randn(B, n_q, H, D, device="cuda", generator=g).half()
    for c in layers:
        c.use_lengths(shared)
        got = c.attend(q, flags=kvc.DETERMINISTIC)
        c.use_lengths(None)
        c.set_lengths(kv_len=kv_len)
        assert torch.equal(got, c.attend(q, flags=kvc.DETERMINISTIC))
    c = layers[-1]
    for b in range(B):
        n = int(kv_len[b])
        assert_close(got[b], orc.attend(to64(q[b]), to64(c.k_store[b, :n]), to64(c.v_store[b, :n])), f"row {b}")


def test_shared_layout_errors_reach_every_user_and_keep_the_last_good_lengths():
    H, D, cap = 4, 128, 256
    layers, g = packed_layers(2, (100, 50), H, D, torch.bfloat16, cap, 9)
    shared = kvc.KVLengths(2, "packed", cap)
    good = torch.tensor([0, 100, 150], dtype=torch.int32, device="cuda")
    shared.set(cu_seqlens=good)
    for c in layers:
        c.use_lengths(shared)
    q = torch.randn(2, 40, H, D, device="cuda", generator=g).bfloat16()
    before = layers[0].attend(q)
    shared.set(cu_seqlens=torch.tensor([0, 100, 300], dtype=torch.int32, device="cuda"))   # past capacity
    assert layers[0].get_error() == kvc.DEV_BAD_CUSEQ
    assert layers[1].get_error() == 0                  # reported once, then cleared
    assert torch.equal(layers[0].attend(q), before)    # the layout kept its last good lengths
    assert layers[0].get_error() == 0


def test_use_lengths_refuses_mismatched_layouts():
    c = kvc.KVCache(2, 4, 4, 128, torch.bfloat16, "packed", capacity=256)
    with pytest.raises(kvc.KvcError) as e:
        c.use_lengths(kvc.KVLengths(3, "packed", 256))                 # another batch
    assert e.value.code == kvc.ERR_ARG
    with pytest.raises(kvc.KvcError) as e:
        c.use_lengths(kvc.KVLengths(2, "packed", 512))                 # more than the store holds
    assert e.value.code == kvc.ERR_ARG
    with pytest.raises(kvc.KvcError) as e:
        c.use_lengths(kvc.KVLengths(2, "linear", 256))                 # another layout
    assert e.value.code == kvc.ERR_UNSUPPORTED
    ring = kvc.KVCache(1, 4, 4, 128, torch.bfloat16, "circular", sink=8, window=32, chunk=8)
    with pytest.raises(kvc.KvcError):
        ring.use_lengths(kvc.KVLengths(1, "linear", 32))


def test_graph_of_one_set_and_many_layers_replays():
    """One captured step: set the shared layout from a device array, then four layers
    attend.  Replays with new lengths copied into that array match eager calls."""
    H, D, cap, n_q = 8, 128, 1024, 128
    layers, g = packed_layers(4, (300, 200), H, D, torch.bfloat16, cap, 13)
    shared = kvc.KVLengths(2, "packed", cap)
    cu = torch.tensor([0, 300, 500], dtype=torch.int32, device="cuda")
    shared.set(cu_seqlens=cu)
    for c in layers:
        c.use_lengths(shared)
    q = torch.randn(2, n_q, H, D, device="cuda", generator=g).bfloat16()
    outs = [torch.empty_like(q) for _ in layers]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            shared.set(cu_seqlens=cu, stream=s)
            for c, o in zip(layers, outs):
                c.attend(q, out=o, stream=s)
    for lens in ((300, 200), (17, 900), (1000, 24)):
        cu.copy_(torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32))
        q.normal_(generator=g)
        graph.replay()
        torch.cuda.synchronize()
        shared.set(cu_seqlens=cu)
        for c, o in zip(layers, outs):
            assert torch.equal(o, c.attend(q)), f"lens {lens}"
    assert layers[0].get_error() == 0
