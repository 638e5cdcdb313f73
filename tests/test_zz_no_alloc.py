"""dsi_indexed_attention_static against dsi_indexed_attention, through the C ABI.

The static entry point serves callers that cannot allocate device memory (a
plugin whose host runtime owns every allocation and gives it no scratch, or a
path that cannot take cudaMalloc's implicit synchronisation): its scratch is a
fixed array inside the library.  This file is collected last so that a run
stopping at its first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from indexed_sparse_attention_indexer_gb300 import binding
from indexed_sparse_attention_indexer_gb300 import workloads as W
from tests.parity import assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _static(lib, g, out, lse, idx, count):
    cache = binding.Cache.of(g)
    st = lib.dsi_indexed_attention_static(
        binding._ptr(g.q_idx), binding._ptr(g.w), binding._ptr(g.q), cache.ref(), g.T, g.H_i,
        g.H, g.K, g.q_offset, g.scale, int(g.mode == "decode"), binding._ptr(idx),
        binding._ptr(count), binding._ptr(out), binding._ptr(lse),
        binding._stream(None))
    return st


def _alloc(g):
    out = torch.empty((g.T, g.H, W.D_LATENT), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((g.T, g.H), dtype=torch.float32, device=DEV)
    idx = torch.empty((g.T, g.K), dtype=torch.int32, device=DEV)
    count = torch.empty((g.T,), dtype=torch.int32, device=DEV)
    return out, lse, idx, count


CASES = {
    "decode_small_heads": lambda: W.make_decode(3, 700, 4, 64, 64, 16, seed=21,
                                                lengths=[700, 33, 410]),
    "decode_hi64_paged_fp8": lambda: W.make_decode(4, 0, 64, 128, 256, 128, seed=22,
                                                   lengths=[3000, 700, 64, 1500], page_size=64,
                                                   k_fp8=True),
    "prefill_hi64": lambda: W.make_prefill(96, 400, 64, 128, 128, 128, seed=23, q_offset=304),
    # 2304 x 2304 fp32 scores alone would be 21 MB: the fused indexer writes
    # none, so the call fits the 16 MiB scratch
    "prefill_scores_beyond_scratch": lambda: W.make_prefill(2304, 2304, 64, 128, 256, 128,
                                                            seed=25),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_matches_workspace_entry_point(name):
    lib = binding.load()
    g = CASES[name]().to(DEV)
    ref_out, ref_lse, ref_idx, ref_cnt = binding.layer(g)
    torch.cuda.synchronize()
    for call in range(2):          # two calls in a row share (and reuse) the scratch
        out, lse, idx, count = _alloc(g)
        st = _static(lib, g, out, lse, idx, count)
        assert st == binding.DSI_OK, lib.dsi_status_string(st)
        torch.cuda.synchronize()
        assert binding.device_status() == 0
        assert torch.equal(idx, ref_idx), f"call {call}: indices differ"
        assert torch.equal(count, ref_cnt)
        assert_out_close(out.float().cpu().numpy(), ref_out.float().cpu().numpy(), f"call {call}")
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        assert float((lse[fin] - ref_lse[fin]).abs().max()) <= 1e-3


def test_static_sizes_prefill_without_score_rows():
    lib = binding.load()
    g = CASES["prefill_scores_beyond_scratch"]().to(DEV)
    cache = binding.Cache.of(g)
    upper = binding.workspace_size(g.T, g.H_i, g.H, g.K, g.T, False)
    exact = binding.layer_workspace_size(cache, g.T, g.H_i, g.H, g.K, 0, False)
    assert upper > (16 << 20) >= exact
    assert exact < g.T * g.T * 4


def test_static_rejects_sizes_beyond_the_scratch():
    lib = binding.load()
    # 64 rows x 65536 score columns x 4 bytes = 16 MiB of scores alone: over the limit
    g = W.make_decode(64, 65536, 4, 64, 8, 16, seed=24).to(DEV)
    out, lse, idx, count = _alloc(g)
    need = binding.workspace_size(g.T, g.H_i, g.H, g.K, g.s_max, True)
    assert need > (16 << 20)
    assert _static(lib, g, out, lse, idx, count) == binding.DSI_ERR_WORKSPACE
