"""The fused layer recorded once into a CUDA graph and replayed.

The C-ABI calls allocate nothing, synchronise nothing and launch only on the
caller's stream (their kernels chained by programmatic stream serialisation),
so a whole decode step or prefill can be captured; a replay with new per-step
inputs in the same buffers must give exactly what a direct call gives (the
kernels are deterministic).
"""
import pytest
import torch

from indexed_sparse_attention_indexer_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _outputs(ws, decode):
    rows = ws.T
    return (torch.empty((rows, ws.H, W.D_LATENT), dtype=torch.bfloat16, device=DEV),
            torch.empty((rows, ws.H), dtype=torch.float32, device=DEV),
            torch.empty((rows, ws.K), dtype=torch.int32, device=DEV),
            torch.empty((rows,), dtype=torch.int32, device=DEV))


def _captured_matches_direct(ws, ws_next, decode):
    """Capture the layer on ws's inputs, replay it on ws_next's per-step
    inputs (same cache), and compare with a direct call on those inputs."""
    cache = binding.Cache.of(ws)
    wsp = binding.alloc_workspace(
        binding.layer_workspace_size(cache, ws.T, ws.H_i, ws.H, ws.K, ws.q_offset, decode), DEV)
    q_idx, w, q = ws.q_idx.clone(), ws.w.clone(), ws.q.clone()
    out, lse, idx, count = _outputs(ws, decode)

    def call():
        binding.indexed_attention(q_idx, w, q, cache, ws.K, ws.scale, decode, ws.q_offset,
                                  out=out, lse=lse, idx=idx, count=count, workspace=wsp)

    call()                        # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    q_idx.copy_(ws_next.q_idx)
    w.copy_(ws_next.w)
    q.copy_(ws_next.q)
    graph.replay()
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    ref = binding.indexed_attention(ws_next.q_idx, ws_next.w, ws_next.q, cache, ws.K, ws.scale,
                                    decode, ws.q_offset)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref[2]) and torch.equal(count, ref[3])
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    # a second replay on the same inputs changes nothing
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(idx, ref[2])


def test_decode_layer_replays_in_a_cuda_graph():
    lens = [3000, 1200, 64, 2500]
    ws = W.make_decode(4, 3000, 64, 128, 256, 128, seed=3, device=DEV, lengths=lens)
    nxt = W.make_decode(4, 3000, 64, 128, 256, 128, seed=4, device=DEV, lengths=lens)
    _captured_matches_direct(ws, nxt, True)


def test_paged_fp8_decode_layer_replays_in_a_cuda_graph():
    lens = [1100, 300, 65]
    ws = W.make_decode(3, 1100, 64, 128, 128, 128, seed=5, device=DEV, lengths=lens, page_size=64,
                       k_fp8=True)
    nxt = W.make_decode(3, 1100, 64, 128, 128, 128, seed=6, device=DEV, lengths=lens,
                        page_size=64, k_fp8=True)
    _captured_matches_direct(ws, nxt, True)


def test_prefill_layer_replays_in_a_cuda_graph():
    ws = W.make_prefill(300, 700, 64, 128, 128, 128, seed=7, device=DEV, q_offset=400)
    nxt = W.make_prefill(300, 700, 64, 128, 128, 128, seed=8, device=DEV, q_offset=400)
    _captured_matches_direct(ws, nxt, False)
