"""The entry points under CUDA graph capture: a serving loop captures its launch-bound
decode steps (and may capture prefill) once and replays them. Every entry point launches
only stream-ordered work on the caller's stream (no allocation, no synchronisation), so a
captured call must give the bits of the same call made directly."""
import pytest
import torch

from linear_attention_serving_02_gb300 import inputs, kda

pytestmark = pytest.mark.gpu


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _capture(fn):
    """Warm up fn on a side stream (first-call set-up stays out of the capture), then
    capture it into a CUDA graph; returns the graph and the outputs of the capture."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


@pytest.mark.parametrize("N,H,steps", [(1, 12, 16), (256, 96, 4)])
def test_decode_steps_replayed_from_a_graph_are_bit_identical(N, H, steps):
    """steps decode calls captured once and replayed, against the same calls made
    directly: outputs and the state updated in place, bit for bit. (1, 12) is the
    launch-bound case a serving loop captures (quarter-row launch); (256, 96) whole rows."""
    S0 = inputs.decode_state(N, H, seed=3, device="cuda")
    toks = [_cuda(inputs.decode_step_inputs(N, H, seed=3, step=i)) for i in range(steps)]
    o_static = [torch.empty((N, H, 128), dtype=torch.float32, device="cuda") for _ in range(steps)]

    eager_state = S0.clone()
    eager = []
    for t in toks:
        eager.append(kda.kda_recurrent_decode(t["q"], t["k"], t["v"], t["z"], t["A"], t["b"], eager_state))
    torch.cuda.synchronize()

    state = S0.clone()

    def run():
        for t, o in zip(toks, o_static):
            kda.kda_recurrent_decode(t["q"], t["k"], t["v"], t["z"], t["A"], t["b"], state, o=o)
        return o_static

    g, _ = _capture(run)  # the warm-up ran the steps once on `state`: start again from S0
    state.copy_(S0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(state, eager_state)
    for a, b in zip(o_static, eager):
        assert torch.equal(a, b)
    # a second replay continues from the state the first one left, like the eager calls would
    for t in toks:
        kda.kda_recurrent_decode(t["q"], t["k"], t["v"], t["z"], t["A"], t["b"], eager_state)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(state, eager_state)


@pytest.mark.parametrize("T,H,n", [(4096, 4, 1), (8192, 12, 1), (30720, 5, 3)])
def test_prefill_replayed_from_a_graph_is_bit_identical(T, H, n):
    """One prefill call captured and replayed: the plain walk (4096 x 4), the segmented walk
    in its chained form (8192 x 12) and with the combine kernel (3 sequences x 5 heads),
    each with its programmatic launch dependencies captured as graph edges."""
    if n == 1:
        cu = cu_h = None
    else:
        cu_h = torch.tensor([0, 10240, 20240, 30720], dtype=torch.int32)
        cu = cu_h.cuda()
    inp = _cuda(inputs.prefill_inputs(T, H, n, seed=11, init_state=True))
    o_ref, S_ref = kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                                         initial_state=inp["S0"], cu_seqlens=cu, cu_seqlens_host=cu_h)
    torch.cuda.synchronize()
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, n, H), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(o_ref)
    S = torch.empty_like(S_ref)

    def run():
        return kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                                     initial_state=inp["S0"], cu_seqlens=cu, cu_seqlens_host=cu_h, o=o,
                                     final_state=S, workspace=ws)

    g, _ = _capture(run)
    o.fill_(float("nan"))
    S.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
    assert kda.kda_workspace_status(ws) == 0
