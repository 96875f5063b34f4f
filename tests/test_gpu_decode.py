"""Recurrent decode on the GPU against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_02_gb300 import inputs, kda
from tests.gpu_util import DECODE_TOL, max_over_rms, np64, rel_frob

pytestmark = pytest.mark.gpu


def _to(d, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _oracle_steps(steps, S0):
    """Decode steps on the oracle: each (n, h) is a sequence fed one token per step."""
    S = np64(S0)
    outs = []
    for st in steps:
        N, H = st["q"].shape[:2]
        o, S = oracle.kda_forward(st["q"].reshape(N, 1, H, 128), st["k"].reshape(N, 1, H, 128),
                                  st["v"].reshape(N, 1, H, 128), st["z"].reshape(N, 1, H, 128), st["A"],
                                  st["b"].reshape(N, 1, H), S0=S)
        outs.append(o[:, 0])
    return outs, S


@pytest.mark.parametrize("N,H", [(3, 2), (1, 12), (80, 8)])
def test_decode_matches_oracle(N, H):
    # (1, 12) and (3, 2) take the quarter-row launch; (80, 8) has 640 >= 4 * 152 pairs: whole rows
    S0 = inputs.decode_state(N, H, seed=1)
    steps = [inputs.decode_step_inputs(N, H, seed=1, step=i) for i in range(6)]
    state = S0.cuda()
    for i, st in enumerate(steps):
        g = _to(st, "cuda")
        o = kda.kda_recurrent_decode(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state)
        torch.cuda.synchronize()
        o_ref, S_ref = _oracle_steps(steps[:i + 1], S0)
        assert max_over_rms(o, o_ref[-1]) <= DECODE_TOL, "step %d o" % i
        assert rel_frob(state, S_ref) <= DECODE_TOL, "step %d state" % i


def test_decode_no_decay_no_write_keeps_state_exactly():
    N, H = 5, 3
    S0 = inputs.decode_state(N, H, seed=2)
    st = inputs.decode_step_inputs(N, H, seed=2)
    st["z"] = torch.full_like(st["z"], -float("inf"))  # a = 1
    st["b"] = torch.full_like(st["b"], -float("inf"))  # beta = 0
    g = _to(st, "cuda")
    state = S0.cuda()
    o = kda.kda_recurrent_decode(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state)
    assert torch.equal(state.cpu(), S0), "a = 1 and beta = 0 must leave the state bit-identical"
    o_ref = np.einsum("nhcj,nhc->nhj", np64(S0), np64(st["q"]))
    assert max_over_rms(o, o_ref) <= DECODE_TOL


def test_decode_full_write_retrieves_value():
    """beta = 1: S_t^T k_t = v_t up to the key's norm (|k| = 1 only to bf16 rounding),
    so compare the retrieval with the oracle's."""
    N, H = 4, 2
    S0 = inputs.decode_state(N, H, seed=3)
    st = inputs.decode_step_inputs(N, H, seed=3)
    st["b"] = torch.full_like(st["b"], float("inf"))
    g = _to(st, "cuda")
    state = S0.cuda()
    kda.kda_recurrent_decode(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state)
    _, S_ref = _oracle_steps([st], S0)
    got = np.einsum("nhcj,nhc->nhj", np64(state), np64(st["k"]))
    ref = np.einsum("nhcj,nhc->nhj", S_ref, np64(st["k"]))
    assert max_over_rms(got, ref) <= DECODE_TOL
    assert max_over_rms(ref, np64(st["v"])) < 2e-2  # close to v itself, to the bf16 norm error


def test_decode_batched_config_sampled():
    """256 sequences x 96 heads, 64 consecutive steps on a 1.6 GB state; the oracle
    follows a sample of (sequence, head) pairs through all steps. Each sampled pair is
    one 'head' of a single-sequence oracle call, so each keeps its own A_h."""
    N, H, steps = 256, 96, 64
    gen = torch.Generator(device="cpu").manual_seed(5)
    pairs = sorted(set((int(n), int(h)) for n, h in zip(torch.randint(0, N, (48,), generator=gen),
                                                        torch.randint(0, H, (48,), generator=gen))))
    P = len(pairs)
    ns = torch.tensor([p[0] for p in pairs])
    hs = torch.tensor([p[1] for p in pairs])
    S0 = inputs.decode_state(N, H, seed=0)
    state = S0.cuda()
    S_s = np64(S0[ns, hs]).reshape(1, P, 128, 128)
    for i in range(steps):
        st = inputs.decode_step_inputs(N, H, seed=0, step=i)
        g = _to(st, "cuda")
        o = kda.kda_recurrent_decode(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state)
        o_ref, S_s = oracle.kda_forward(st["q"][ns, hs].reshape(1, 1, P, 128), st["k"][ns, hs].reshape(1, 1, P, 128),
                                        st["v"][ns, hs].reshape(1, 1, P, 128), st["z"][ns, hs].reshape(1, 1, P, 128),
                                        st["A"][hs].contiguous(), st["b"][ns, hs].reshape(1, 1, P), S0=S_s)
        assert max_over_rms(o[ns, hs].cpu(), o_ref[0, 0]) <= DECODE_TOL, "step %d o" % i
    torch.cuda.synchronize()
    assert rel_frob(state[ns, hs], S_s[0]) <= DECODE_TOL
    assert torch.isfinite(state).all()


@pytest.mark.parametrize("extra", [-1, 0])
def test_decode_at_the_column_split_boundary(extra):
    """Just below and at the pair count where decode switches from quarter-row CTAs to
    whole-row CTAs (four per SM of this device): both against the oracle, and verify and
    fold (which must take the same split) bit for bit against it."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = 4 * sms + extra
    N, H = pairs, 1
    steps = [inputs.decode_step_inputs(N, H, seed=31, step=t) for t in range(2)]
    S0 = inputs.decode_state(N, H, seed=31)
    state = S0.cuda()
    outs = []
    for st in steps:
        g = _to(st, "cuda")
        outs.append(kda.kda_recurrent_decode(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], state))
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle_steps(steps, S0)
    for t in range(2):
        assert max_over_rms(outs[t], o_ref[t]) <= DECODE_TOL, t
    assert rel_frob(state, S_ref) <= DECODE_TOL
    # verify over the same two tokens from the checkpoint, then fold both: identical bits
    win = {key: torch.stack([st[key] for st in steps], 1).reshape((N * 2,) + tuple(steps[0][key].shape[1:]))
           for key in ("q", "k", "v", "z", "b")}
    g = _to(win, "cuda")
    S0c = S0.cuda()
    o_v, gk, beta = kda.kda_recurrent_verify(g["q"], g["k"], g["v"], g["z"], steps[0]["A"].cuda(), g["b"], S0c, 2)
    o_v = o_v.reshape(N, 2, H, 128)
    for t in range(2):
        assert torch.equal(o_v[:, t], outs[t]), t
    acc = torch.full((N,), 2, dtype=torch.int32, device="cuda")
    folded = S0c.clone()
    kda.kda_replay_fold(g["k"], g["v"], gk, beta, acc, folded, 2)
    assert torch.equal(folded, state)


def test_decode_writes_every_output_over_poison():
    """o starts as NaN: every (sequence, head, channel) is written."""
    for N, H in ((3, 2), (80, 8)):  # quarter-row and whole-row launches
        st = _to(inputs.decode_step_inputs(N, H, seed=41, step=0), "cuda")
        state = inputs.decode_state(N, H, seed=41).cuda()
        o = torch.full((N, H, 128), float("nan"), dtype=torch.float32, device="cuda")
        kda.kda_recurrent_decode(st["q"], st["k"], st["v"], st["z"], st["A"], st["b"], state, o=o)
        torch.cuda.synchronize()
        assert torch.isfinite(o).all() and torch.isfinite(state).all()
