"""The prefill entry point that allocates nothing.

Some callers of this library cannot allocate device memory: a plugin inside an engine
that owns all of the GPU's memory and hands it only the tensors of each call, or code on
a latency-critical path where cudaMalloc may stall the whole device. They call
kda_chunk_prefill_noalloc, which runs the same kernels on a fixed scratch area built
into the library instead of a caller workspace. This file checks, through the C ABI,
that it gives, bit for bit, what kda_chunk_prefill gives on two calls in a row (the
second call must not see anything the first left in the shared scratch; both run the
same kernels with the same launch shapes, so any stale value would show), that a bad
device cu_seqlens marks the final states invalid and leaves the next call exact, that
the binding rejects malformed inputs, and that a batch too large for the scratch is
refused before anything runs. It is named to run after every other test
file, and it passes alone in a fresh process as well.
"""
import ctypes

import pytest
import torch

from linear_attention_serving_02_gb300 import inputs, kda

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
    assert torch.equal(o_na, o_ref) and torch.equal(S_na, S_ref)
    # second call right after, on a different batch shape and different inputs
    second = inputs.prefill_inputs(2 * 200, 3, 2, seed=32, init_state=True, batch_rows=2)
    (o_ref, S_ref), (o_na, S_na) = _both(second)
    assert torch.equal(o_na, o_ref) and torch.equal(S_na, S_ref)


def test_noalloc_bad_device_cu_seqlens_then_a_good_call():
    """A falling cu_seqlens with no host copy is caught on the device: every final state
    comes back NaN and o is left alone. The next call on the same scratch is exact."""
    H = 2
    g = _cuda(inputs.prefill_inputs(256, H, 3, seed=33, init_state=True))
    o = torch.full(g["q"].shape, 7.0, dtype=torch.float32, device="cuda")
    bad = torch.tensor([0, 100, 50, 256], dtype=torch.int32, device="cuda")
    _, S = kda.kda_chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=g["S0"],
                                         cu_seqlens=bad, o=o)
    torch.cuda.synchronize()
    assert torch.isnan(S).all()
    assert (o == 7.0).all()
    (o_ref, S_ref), (o_na, S_na) = _both(inputs.prefill_inputs(256, H, 3, seed=34, init_state=True), [0, 50, 100, 256])
    assert torch.equal(o_na, o_ref) and torch.equal(S_na, S_ref)


def test_noalloc_binding_rejects_malformed_inputs():
    """The binding checks what the C ABI cannot see: a cu_seqlens_host that lives on the
    device, or has the wrong length, and a dense batch whose q is not [B, T, H, 128]."""
    g = _cuda(inputs.prefill_inputs(128, 2, 2, seed=35))
    cu = torch.tensor([0, 64, 128], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        kda.kda_chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], cu_seqlens=cu,
                                      cu_seqlens_host=cu)
    with pytest.raises(ValueError):
        kda.kda_chunk_prefill_noalloc(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], cu_seqlens=cu,
                                      cu_seqlens_host=torch.tensor([0, 128], dtype=torch.int32))
    q3 = g["q"][0]
    with pytest.raises(ValueError):
        kda.kda_chunk_prefill_noalloc(q3, g["k"][0], g["v"][0], g["z"][0], g["A"], g["b"][0])


def test_noalloc_refuses_a_batch_larger_than_its_scratch():
    lib = kda.library()
    fn = lib.kda_chunk_prefill_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp, vp]
    fn.restype = ctypes.c_int
    fake = 1 << 20  # never dereferenced: the size check refuses the call before any launch
    rc = fn(fake, fake, fake, fake, fake, fake, None, None, None, 1, 1 << 20, 1, 12, 128, 128, fake, 0, fake, None)
    assert rc == KDA_ERR_WORKSPACE
