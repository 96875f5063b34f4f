"""The prefill entry point that allocates nothing.

Some callers of this library cannot allocate device memory: a plugin inside an engine
that owns all of the GPU's memory and hands it only the tensors of each call, or code on
a latency-critical path where cudaMalloc may stall the whole device. They call
kda_chunk_prefill_noalloc, which runs the same kernels on a fixed scratch area built
into the library instead of a caller workspace. This file checks, through the C ABI,
that it gives what kda_chunk_prefill gives on two calls in a row (the second call must
not see anything the first left in the shared scratch), and that a batch too large for
the scratch is refused before anything runs. It is named to run after every other test
file, and it passes alone in a fresh process as well.
"""
import ctypes

import pytest
import torch

from linear_attention_serving_02_gb300 import inputs, kda
from tests.gpu_util import PREFILL_O_TOL, PREFILL_S_TOL, max_over_rms, rel_frob

pytestmark = pytest.mark.gpu

KDA_ERR_WORKSPACE = -6


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _both(inp, cu=None):
    g = _cuda(inp)
    cu_d = None if cu is None else torch.tensor(cu, dtype=torch.int32, device="cuda")
    ref = kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=g["S0"],
                                cu_seqlens=cu_d, o_dtype=torch.float32)
    got = kda.kda_chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=g["S0"],
                                        cu_seqlens=cu_d, o_dtype=torch.float32)
    torch.cuda.synchronize()
    return [t.cpu() for t in ref], [t.cpu() for t in got]


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # first call: packed varlen batch with an empty sequence and a partial last chunk
    lens = [300, 0, 64, 700]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    first = inputs.prefill_inputs(cu[-1], 4, len(lens), seed=31, init_state=True)
    (o_ref, S_ref), (o_na, S_na) = _both(first, cu)
    assert max_over_rms(o_na, o_ref) <= PREFILL_O_TOL
    assert rel_frob(S_na, S_ref) <= PREFILL_S_TOL
    # second call right after, on a different batch shape and different inputs
    second = inputs.prefill_inputs(2 * 200, 3, 2, seed=32, init_state=True, batch_rows=2)
    (o_ref, S_ref), (o_na, S_na) = _both(second)
    assert max_over_rms(o_na, o_ref) <= PREFILL_O_TOL
    assert rel_frob(S_na, S_ref) <= PREFILL_S_TOL


def test_noalloc_refuses_a_batch_larger_than_its_scratch():
    lib = kda.library()
    fn = lib.kda_chunk_prefill_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp, vp]
    fn.restype = ctypes.c_int
    fake = 1 << 20  # never dereferenced: the size check refuses the call before any launch
    rc = fn(fake, fake, fake, fake, fake, fake, None, None, None, 1, 1 << 20, 1, 12, 128, 128, fake, 0, fake, None)
    assert rc == KDA_ERR_WORKSPACE
