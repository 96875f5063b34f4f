"""The state walk's failure path, made to happen without a GPU fault: a host-set hook
makes the walk's MMA issuer leave out one chunk's (or one chained map's) completion
signal, so the waits behind it run out (after a shortened limit) while every MMA still
completes. The walk must then
report KDA_ERR_CUDA through the workspace status word, fill its final state with NaN,
leave the context usable, and a clean call afterwards must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_02_gb300 import inputs, kda
from tests.gpu_util import assert_prefill_close

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 2_000_000_000


def _cuda(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


@pytest.mark.parametrize("T,skip", [
    (192, 1),     # the plain walk: chunk slot 1's group-1 signal
    (4096, 1),    # the segmented walk (one long sequence, 11 segments of 6 chunks)
    (4096, -2),   # ... the first map of the output walks' map chain
    (4096, -5),   # ... its fourth map (only the segments with at least four maps fail)
])
def test_walk_wait_runs_out_and_is_reported(T, skip):
    H = 2
    inp_cpu = inputs.prefill_inputs(T, H, 1, seed=41, init_state=True)
    inp = _cuda(inp_cpu)
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, 1, H), dtype=torch.uint8, device="cuda")
    o = torch.empty(inp["q"].shape, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    if skip < 0:  # the map chain runs only in the chained segmented form
        assert kda.kda_chunk_prefill_walk_form(T, 1, H) == 1
    kda.kda_debug_walk_fault(skip, 1_000_000)  # waits give up after 1 ms
    try:
        _, S = kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                                     initial_state=inp["S0"], o=o, workspace=ws, o_dtype=torch.float32)
        torch.cuda.synchronize()
        status = kda.kda_workspace_status(ws)
    finally:
        kda.kda_debug_walk_fault(-1, DEFAULT_LIMIT_NS)
    assert status == -7, status
    assert torch.isnan(S).all(), "the failed walks' final states must be NaN"
    # the context is usable, and the same workspace serves a clean call that is correct
    _, S2 = kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                                  initial_state=inp["S0"], o=o, workspace=ws, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_workspace_status(ws) == 0
    o_ref, S_ref = oracle.kda_forward(inp_cpu["q"], inp_cpu["k"], inp_cpu["v"], inp_cpu["z"], inp_cpu["A"],
                                      inp_cpu["b"], S0=inp_cpu["S0"])
    assert_prefill_close(o.cpu(), S2.cpu(), o_ref, S_ref, "after the failed call")


def test_fault_hook_rejects_a_zero_limit():
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_debug_walk_fault(-1, 0)
    assert ei.value.status == -2
