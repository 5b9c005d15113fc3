"""The streaming DiT workload at full size with each chunk's lifecycle captured as one
CUDA graph: reserve the chunk's slots, then four denoising rewrites, each a write of the
chunk's K/V at the device-held slots and an attend of its queries over the sink+window
ring (flashdreams issue "add an opt-in circular KV policy for streaming attention",
"proposed boundary": reservation separate from writes, device-resident write metadata, so
a captured step writes the slot the device holds on every replay).  Replayed over the 10
chunks (7 fill the 32760-slot ring, 3 evict), it equals the eager run bit for bit.
"""
import pytest
import torch

from diffusion_serving_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from diffusion_serving_gb300 import kvc


def bits(t):
    return t.view(torch.int16)


def test_dit_chunk_graph_replays_equal_the_eager_run():
    w = wl.DIT_STREAM
    R = w.rewrites
    mk = lambda: kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.bfloat16, "circular",
                             sink=w.sink, window=w.window, chunk=w.chunk)
    eager, cache = mk(), mk()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    bufs = [tuple(torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in (
        (w.batch, w.chunk, w.heads, w.head_dim), (w.batch, w.chunk, w.kv_heads, w.head_dim),
        (w.batch, w.chunk, w.kv_heads, w.head_dim))) for _ in range(R)]
    outs = [torch.empty_like(bufs[0][0]) for _ in range(R)]

    def chunk_body(stream):
        cache.advance(stream=stream)
        for (q, k, v), o in zip(bufs, outs):
            cache.write(k, v, stream=stream)
            cache.attend(q, o, stream=stream)

    def load(c):
        for r in range(R):
            for dst, src in zip(bufs[r], wl.chunk_inputs(w, c, r, device="cuda")):
                dst.copy_(src)

    graph = torch.cuda.CUDAGraph()
    bases = []
    for c in range(w.n_chunks):
        load(c)
        torch.cuda.synchronize()
        if c == 0:                                      # chunk 0 eager, then capture the chunk
            with torch.cuda.stream(side):
                chunk_body(side)
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                chunk_body(side)
        else:
            graph.replay()
        torch.cuda.synchronize()
        bases.append(cache.row_state()[0][1])
        eager.advance()
        for r, (q, k, v) in enumerate(bufs):
            eager.write(k, v)
            want = eager.attend(q)
            assert torch.equal(bits(outs[r]), bits(want)), f"chunk {c} rewrite {r}"
    assert bases == [c * w.chunk for c in range(7)] + [w.sink + i * w.chunk for i in range(3)]
    assert torch.equal(bits(cache.k_store), bits(eager.k_store))
    assert torch.equal(bits(cache.v_store), bits(eager.v_store))
    assert cache.get_error() == 0 and eager.get_error() == 0
