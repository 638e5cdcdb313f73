"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes runs out, the kernel reports DSI_ERR_TIMEOUT through the device
status word and ends, and the context stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import oracle
from indexed_sparse_attention_indexer_gb300 import binding
from indexed_sparse_attention_indexer_gb300 import workloads as W
from tests.parity import assert_out_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("checked", [False, True], ids=["release", "checked"])
def test_bounded_wait_times_out_and_the_context_survives(checked):
    assert binding.device_status(checked=checked) == binding.DSI_OK     # nothing pending
    t0 = time.perf_counter()
    binding.selftest_wait_timeout(1_000_000, checked=checked)          # a 1 ms limit
    st = binding.device_status(checked=checked)                        # synchronises
    elapsed = time.perf_counter() - t0
    assert st == binding.DSI_ERR_TIMEOUT
    assert elapsed < 1.0, f"the wait should give up after ~1 ms, took {elapsed:.3f} s"
    assert binding.device_status(checked=checked) == binding.DSI_OK     # read once, then cleared
    # the next call of the layer runs clean and right
    ws = W.make_decode(2, 0, 64, 128, 64, 128, seed=41, lengths=[900, 130])
    g = ws.to("cuda")
    out, lse, idx, count = binding.layer(g, checked=checked)
    torch.cuda.synchronize()
    assert binding.device_status(checked=checked) == binding.DSI_OK
    ref = oracle.layer(ws)
    for b in range(ws.B):
        assert np.array_equal(idx[b].cpu().numpy(), ref[b]["idx"])
    assert_out_close(out.float().cpu().numpy(), np.stack([ref[b]["out"] for b in range(ws.B)]),
                     "after timeout")
