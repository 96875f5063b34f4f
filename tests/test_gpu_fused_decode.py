"""The fused decode layer step (conv -> recurrent update -> gated RMSNorm) on the GPU,
through the C ABI, against the fp64 oracle of oracle/layer.py. The conv state is byte
work (a shift of bf16 inputs), so it must match bit for bit."""
import numpy as np
import pytest
import torch

from linear_attention_serving_02_gb300 import inputs, kda
from oracle import layer
from tests.gpu_util import DECODE_TOL, max_over_rms, np64, rel_frob

pytestmark = pytest.mark.gpu

EPS_L2, EPS_RMS = 1e-6, 1e-5


def _cuda(d):
    return {k: v.cuda() for k, v in d.items()}


def _run(N, H, steps, seed, conv0=None):
    prm = inputs.fused_decode_params(H, seed=seed)
    S0 = inputs.decode_state(N, H, seed=seed)
    cs0 = torch.zeros((N, 3, 3, H, 128), dtype=torch.bfloat16) if conv0 is None else conv0
    gp = _cuda(prm)
    state, cs = S0.cuda(), cs0.cuda()
    S_ref, cs_ref = np64(S0), cs0.clone()
    for t in range(steps):
        st = inputs.fused_decode_step_inputs(N, H, seed=seed, step=t)
        g = _cuda(st)
        y = kda.kda_fused_decode(g["x_q"], g["x_k"], g["x_v"], cs, gp["conv_w"], g["z"], g["A"], g["b"], g["g"],
                                 gp["norm_w"], state, eps_l2=EPS_L2, eps_rms=EPS_RMS)
        torch.cuda.synchronize()
        y_ref, S_ref, _ = layer.fused_decode(st["x_q"], st["x_k"], st["x_v"], cs_ref, prm["conv_w"], st["z"],
                                             st["A"], st["b"], st["g"], prm["norm_w"], S_ref, EPS_L2, EPS_RMS)
        # the conv state keeps the last three raw inputs of each stream
        cs_ref = torch.cat([cs_ref[:, :, 1:], torch.stack([st["x_q"], st["x_k"], st["x_v"]], 1)[:, :, None]], 2)
        assert torch.equal(cs.cpu(), cs_ref), "conv state at step %d" % t
        assert max_over_rms(y, y_ref) <= DECODE_TOL, "y at step %d" % t
        assert rel_frob(state, S_ref) <= DECODE_TOL, "state at step %d" % t


@pytest.mark.parametrize("N,H", [(3, 2), (1, 12), (80, 8)])
def test_fused_decode_matches_oracle(N, H):
    # (3, 2) and (1, 12): clusters of four quarter-row CTAs; (80, 8): one CTA per head
    _run(N, H, steps=5, seed=21)


@pytest.mark.parametrize("N,H", [(2, 3), (80, 8)])
def test_fused_decode_continues_a_conv_state(N, H):
    g = torch.Generator().manual_seed(3)
    conv0 = torch.randn((N, 3, 3, H, 128), generator=g).to(torch.bfloat16)
    _run(N, H, steps=2, seed=22, conv0=conv0)


def test_fused_decode_full_size_sampled():
    """256 sequences x 96 heads (1.6 GB of state), 3 tokens: y and the state on sampled
    (sequence, head) units against the oracle, the whole conv state bit for bit."""
    N, H, T = 256, 96, 3
    seed = 23
    prm = inputs.fused_decode_params(H, seed=seed)
    gp = _cuda(prm)
    S0 = inputs.decode_state(N, H, seed=seed)
    state = S0.cuda()
    cs = torch.zeros((N, 3, 3, H, 128), dtype=torch.bfloat16, device="cuda")
    steps = [inputs.fused_decode_step_inputs(N, H, seed=seed, step=t) for t in range(T)]
    ys = []
    for st in steps:
        g = _cuda(st)
        ys.append(kda.kda_fused_decode(g["x_q"], g["x_k"], g["x_v"], cs, gp["conv_w"], g["z"], g["A"], g["b"],
                                       g["g"], gp["norm_w"], state, eps_l2=EPS_L2, eps_rms=EPS_RMS).cpu())
    expect = torch.zeros((N, 3, 3, H, 128), dtype=torch.bfloat16)
    for st in steps:
        expect = torch.cat([expect[:, :, 1:], torch.stack([st["x_q"], st["x_k"], st["x_v"]], 1)[:, :, None]], 2)
    assert torch.equal(cs.cpu(), expect)
    state_c = state.cpu()
    for (n, h) in [(0, 0), (77, 5), (255, 95)]:
        S = np64(S0[n:n + 1, h:h + 1])
        c = torch.zeros((1, 3, 3, 1, 128), dtype=torch.bfloat16)
        for t, st in enumerate(steps):
            sl = {k: (v[n:n + 1, h:h + 1] if k != "A" else v[h:h + 1]) for k, v in st.items()}
            y_ref, S, c_new = layer.fused_decode(sl["x_q"], sl["x_k"], sl["x_v"], c, prm["conv_w"][:, h:h + 1],
                                                 sl["z"], sl["A"], sl["b"], sl["g"], prm["norm_w"], S, EPS_L2,
                                                 EPS_RMS)
            c = torch.from_numpy(c_new).to(torch.bfloat16)
            assert max_over_rms(ys[t][n, h], y_ref[0, 0]) <= DECODE_TOL, (n, h, t)
        assert rel_frob(state_c[n, h], S[0, 0]) <= DECODE_TOL, (n, h)
