"""Multi-token verify and the ReplaySSM fold on the GPU, through the C ABI: against the
fp64 oracle, and bit for bit against repeated single-token decode calls (the property
'Kimi K3 attention deep dive', §6.2, asks of the fold)."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_02_gb300 import inputs, kda
from tests.gpu_util import DECODE_TOL, max_over_rms, np64, rel_frob

pytestmark = pytest.mark.gpu


def _window(N, H, m, seed):
    """m decode steps of N sequences stacked token-major: token t of sequence n at row n*m+t."""
    steps = [inputs.decode_step_inputs(N, H, seed=seed, step=t) for t in range(m)]
    win = {}
    for key in ("q", "k", "v", "z", "b"):
        x = torch.stack([st[key] for st in steps], dim=1)  # [N, m, H, ...]
        win[key] = x.reshape((N * m,) + tuple(x.shape[2:])).contiguous()
    win["A"] = steps[0]["A"]
    return steps, win


def _cuda(d):
    return {k: v.cuda() for k, v in d.items()}


def _decode_snapshots(steps, S0):
    """The state before and after each of m single-token decode calls, and their outputs."""
    state = S0.clone()
    snaps, outs = [state.clone()], []
    for st in steps:
        g = _cuda(st)
        outs.append(kda.kda_recurrent_decode(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state))
        snaps.append(state.clone())
    return snaps, outs


@pytest.mark.parametrize("N,H,m", [(4, 3, 8), (2, 5, 1), (3, 2, 16), (80, 8, 7)])
def test_verify_matches_oracle(N, H, m):
    steps, win = _window(N, H, m, seed=11)
    S0 = inputs.decode_state(N, H, seed=11)
    g = _cuda(win)
    state = S0.cuda()
    state_out = torch.empty_like(state)
    o, gk, beta = kda.kda_recurrent_verify(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state, m,
                                           state_out=state_out)
    torch.cuda.synchronize()
    assert torch.equal(state.cpu(), S0), "verify must not write the checkpoint"
    o_ref, S_ref, la_ref, beta_ref = oracle.verify(win["q"], win["k"], win["v"], win["z"], win["A"], win["b"],
                                                   S0, m)
    assert max_over_rms(o, o_ref) <= DECODE_TOL
    assert rel_frob(state_out, S_ref) <= DECODE_TOL
    # the logged gate values are the fp32 evaluations of the same formulas
    assert np.max(np.abs(np64(gk) - la_ref)) <= 4e-6
    assert np.max(np.abs(np64(beta) - beta_ref)) <= 1e-6


@pytest.mark.parametrize("N,H", [(4, 3), (80, 8)])
def test_verify_and_fold_are_bit_identical_to_decode(N, H):
    # (4, 3): quarter-row launch; (80, 8): 640 >= 4 * 152 pairs, whole rows
    m = 8
    steps, win = _window(N, H, m, seed=12)
    S0 = inputs.decode_state(N, H, seed=12).cuda()
    snaps, outs = _decode_snapshots(steps, S0)
    g = _cuda(win)
    o, gk, beta = kda.kda_recurrent_verify(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], S0, m)
    o = o.reshape(N, m, H, 128)
    for t in range(m):
        assert torch.equal(o[:, t], outs[t]), "verify output of token %d differs from decode" % t
    rng = np.random.default_rng(5)
    for accepted in (rng.integers(0, m + 1, N), np.full(N, m), np.zeros(N, dtype=np.int64),
                     np.array([(-1) ** n * (m + 2 + n) for n in range(N)])):
        acc = torch.tensor(accepted, dtype=torch.int32, device="cuda")
        state = S0.clone()
        kda.kda_replay_fold(g["k"], g["v"], gk, beta, acc, state, m)
        torch.cuda.synchronize()
        for n in range(N):
            a = int(min(max(accepted[n], 0), m))
            assert torch.equal(state[n], snaps[a][n]), "fold of %d tokens (sequence %d)" % (a, n)


def test_multi_token_decode_in_place():
    """state_out = state: m tokens in one call, bit-identical to m decode calls."""
    N, H, m = 6, 4, 5
    steps, win = _window(N, H, m, seed=13)
    S0 = inputs.decode_state(N, H, seed=13).cuda()
    snaps, outs = _decode_snapshots(steps, S0)
    g = _cuda(win)
    state = S0.clone()
    o, gk, beta = kda.kda_recurrent_verify(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state, m,
                                           state_out=state, log=False)
    assert gk is None and beta is None
    assert torch.equal(state, snaps[m])
    assert torch.equal(o.reshape(N, m, H, 128)[:, m - 1], outs[m - 1])


def test_fold_matches_oracle_replay():
    N, H, m = 5, 2, 6
    steps, win = _window(N, H, m, seed=14)
    S0 = inputs.decode_state(N, H, seed=14)
    g = _cuda(win)
    _, gk, beta = kda.kda_recurrent_verify(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], S0.cuda(), m)
    accepted = [0, 6, 3, 1, 5]
    state = S0.cuda()
    kda.kda_replay_fold(g["k"], g["v"], gk, beta, torch.tensor(accepted, dtype=torch.int32, device="cuda"), state, m)
    la_ref, beta_ref = oracle.gate(win["z"], win["A"], win["b"])
    S_ref = oracle.replay_fold(win["k"], win["v"], la_ref, beta_ref, S0, accepted, m)
    for n in range(N):
        if accepted[n] == 0:
            assert torch.equal(state[n].cpu(), S0[n])
        else:
            assert rel_frob(state[n], S_ref[n]) <= DECODE_TOL, "sequence %d" % n


def test_full_size_window():
    """256 sequences x 96 heads, a 7-token draft window (the pages' num_speculative_tokens):
    verify on sampled (sequence, head) units against the oracle, fold bit for bit against
    single-token decode snapshots of the whole 1.6 GB state."""
    N, H, m = 256, 96, 7
    steps, win = _window(N, H, m, seed=15)
    S0 = inputs.decode_state(N, H, seed=15).cuda()
    snaps, outs = _decode_snapshots(steps, S0)
    g = _cuda(win)
    o, gk, beta = kda.kda_recurrent_verify(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], S0, m)
    o4 = o.reshape(N, m, H, 128)
    for t in range(m):
        assert torch.equal(o4[:, t], outs[t]), "token %d" % t
    acc_np = np.random.default_rng(7).integers(0, m + 1, N)
    acc = torch.tensor(acc_np, dtype=torch.int32, device="cuda")
    state = S0.clone()
    kda.kda_replay_fold(g["k"], g["v"], gk, beta, acc, state, m)
    stacked = torch.stack(snaps)  # [m + 1, N, H, 128, 128]
    expect = stacked[torch.tensor(acc_np, device="cuda"), torch.arange(N, device="cuda")]
    assert torch.equal(state, expect)
    del stacked, expect
    # sampled units against the oracle
    S0c = S0.cpu()
    for (n, h) in [(0, 0), (131, 47), (255, 95)]:
        rows = slice(n * m, (n + 1) * m)
        o_ref, _, _, _ = oracle.verify(win["q"][rows, h:h + 1], win["k"][rows, h:h + 1], win["v"][rows, h:h + 1],
                                       win["z"][rows, h:h + 1], win["A"][h:h + 1], win["b"][rows, h:h + 1],
                                       S0c[n:n + 1, h:h + 1], m)
        assert max_over_rms(o4[n, :, h].cpu(), o_ref[:, 0]) <= DECODE_TOL, (n, h)
