"""Prefill at the full workload sizes, in the launch configuration the benchmark times.

- one sequence of 8192 tokens, 12 heads, random initial state: every output compared;
- 8 packed sequences of 1024..32768 tokens, 32 heads: sampled (sequence, head) units;
- one sequence of 1,048,576 tokens, 12 heads, then 128 decode steps: one head followed
  by the oracle end to end, all heads checked against a single prefill of T + 128.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_02_gb300 import inputs, kda
from tests.gpu_util import PREFILL_O_TOL, PREFILL_S_TOL, assert_prefill_close, max_over_rms, np64, oracle_units, rel_frob

pytestmark = pytest.mark.gpu


def test_single_sequence_8192_tokens_12_heads():
    T, H = 8192, 12
    inp = inputs.prefill_inputs(T, H, 1, seed=0, init_state=True)
    g = {k: v.cuda() for k, v in inp.items()}
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    for dt in (torch.bfloat16, torch.float32):
        o, S = kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=g["S0"],
                                     o_dtype=dt)
        torch.cuda.synchronize()
        assert_prefill_close(o.cpu(), S.cpu(), o_ref, S_ref, "T=8192 %s" % dt)


def test_packed_varlen_8_sequences_32_heads_sampled():
    H = 32
    lens = inputs.varlen_lengths(8, 1024, 32768, seed=0)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    inp = inputs.prefill_inputs(cu[-1], H, len(lens), seed=0)
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o, S = kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], cu_seqlens=cu_d,
                                 cu_seqlens_host=torch.tensor(cu, dtype=torch.int32), o_dtype=torch.float32)
    torch.cuda.synchronize()
    del g
    o, S = o.cpu(), S.cpu()
    short, long_ = int(np.argmin(lens)), int(np.argmax(lens))
    units = [(short, 0), (short, 31), (long_, 5), (3, 17), (6, 9)]
    ref = oracle_units(inp, cu, units)
    for (n, h), (o_ref, S_ref) in ref.items():
        assert_prefill_close(o[0, cu[n]:cu[n + 1], h], S[n, h], o_ref, S_ref, "seq %d head %d" % (n, h))
    assert torch.isfinite(o).all() and torch.isfinite(S).all()


def test_million_token_prefill_then_128_decode_steps():
    T, m, H = 1 << 20, 128, 12
    inp = inputs.prefill_inputs(T + m, H, 1, seed=0, device="cuda")   # drawn on the device: 16 GB of inputs
    q, k, v, z, A, b = (inp[x] for x in ("q", "k", "v", "z", "A", "b"))
    # reference run on the GPU: one prefill over all T + m tokens
    o_long, S_long = kda.kda_chunk_prefill(q, k, v, z, A, b, o_dtype=torch.float32)
    torch.cuda.synchronize()
    # prefill the first T tokens, then feed the state to m recurrent decode steps
    head = [x[:, :T] for x in (q, k, v, z, b)]
    o1, S = kda.kda_chunk_prefill(head[0], head[1], head[2], head[3], A, head[4], o_dtype=torch.float32)
    outs = []
    for t in range(T, T + m):
        outs.append(kda.kda_recurrent_decode(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                                             z[:, t].contiguous(), A, b[:, t].contiguous(), S))
    torch.cuda.synchronize()
    o_dec = torch.stack(outs, 0)[:, 0]                                 # [m, H, 128]
    assert torch.isfinite(o1).all() and torch.isfinite(S).all()
    # both paths agree on the final state and on the last m outputs
    assert rel_frob(S.cpu(), S_long.cpu()) <= PREFILL_S_TOL
    assert max_over_rms(o_dec.cpu(), o_long[0, T:].cpu()) <= PREFILL_O_TOL
    assert max_over_rms(o1[0].cpu(), o_long[0, :T].cpu()) <= PREFILL_O_TOL
    # head 3 followed by the oracle over all T + m tokens (column blocks of 8 spread it over the host cores)
    h = 3
    sl = lambda x: x[0, :, h:h + 1].cpu()
    la, beta = oracle.gate(sl(z), A[h:h + 1].cpu(), b[0, :, h:h + 1].cpu())
    o_ref, S_ref = oracle.recurrence(sl(q), sl(k), sl(v), la, beta, col_block=8)
    assert rel_frob(S[0, h].cpu(), S_ref[0, 0]) <= PREFILL_S_TOL
    assert max_over_rms(o_dec[:, h].cpu(), o_ref[T:, 0]) <= PREFILL_O_TOL
    idx = torch.arange(0, T, 997)
    assert max_over_rms(o1[0, idx, h].cpu(), o_ref[idx.numpy(), 0]) <= PREFILL_O_TOL
