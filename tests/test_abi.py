"""The C-ABI library on the CPU: it builds, loads, exports every entry point that
include/*.h declares, and its host-side argument checks return the documented status
codes. No compute call is made here; the checks reject every case before any CUDA
call, so fake (never dereferenced) device pointers are safe to pass.
"""
import ctypes
import glob
import os
import re

import pytest

from linear_attention_serving_02_gb300 import kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KDA_OK, KDA_ERR_NULL, KDA_ERR_SHAPE, KDA_ERR_UNSUPPORTED = 0, -1, -2, -3
KDA_ERR_SEQLENS, KDA_ERR_ALIGN, KDA_ERR_WORKSPACE = -4, -5, -6
FAKE = 1 << 20  # 256-byte aligned fake device address, never dereferenced
KDA_MAX_REPLAY = 16


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(kda_[A-Za-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("kda_chunk_prefill", "kda_recurrent_decode", "kda_chunk_prefill_workspace_size",
                     "kda_status_string", "kda_workspace_status", "kda_version",
                     "kda_chunk_prefill_launch_count", "kda_recurrent_verify", "kda_replay_fold", "kda_fused_decode"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(kda.library()._name)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, "not exported: %s" % missing


def test_status_strings_and_version():
    assert kda.kda_status_string(0) == "ok"
    for code in range(-8, 0):
        assert kda.kda_status_string(code) != "unknown status"
    assert kda.kda_status_string(12345) == "unknown status"
    assert kda.kda_version() >= 100


def test_segment_ends_hook_checks():
    for bad in (-1, 65):
        with pytest.raises(kda.KdaError):
            kda.kda_debug_segment_ends(bad)
    kda.kda_debug_segment_ends(3)
    kda.kda_debug_segment_ends(0)


def test_workspace_size():
    ws = kda.kda_chunk_prefill_workspace_size
    assert ws(-1, 1, 1) == 0
    a = ws(8192, 1, 12)
    b = ws(8192 * 2, 1, 12)
    assert 0 < a < b
    assert ws(8192, 1, 24) > a
    # one more sequence can add a partial chunk per head
    assert ws(8192, 2, 12) > a


def test_launch_count():
    lc = kda.kda_chunk_prefill_launch_count
    assert lc(-1, 1, 1) == -1
    assert lc(0, 0, 4) == 0
    # many (sequence, head) chains fill the GPU: one walk pass
    assert lc(8192 * 64, 64, 32) == 3
    # short chains are not worth splitting
    assert lc(256, 1, 2) == 3
    # one long sequence over few heads: segmented walk (5 launches), every output walk in
    # one wave chaining the maps itself (form 1), or more segments than that and a combine
    # kernel (form 2)
    assert lc(8192, 1, 12) == 5
    assert lc(1 << 20, 1, 12) == 5
    wf = kda.kda_chunk_prefill_walk_form
    assert wf(-1, 1, 1) == -1 and wf(0, 0, 4) == 0
    assert wf(8192 * 64, 64, 32) == 0 and wf(256, 1, 2) == 0
    assert wf(8192, 1, 12) == 1 and wf(1 << 20, 1, 12) == 2


def _prefill(**over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, A=FAKE, b=FAKE, initial_state=None, cu=None, cu_host=None,
                batch=1, seq_len=256, num_seqs=1, num_heads=2, d_k=128, d_v=128, o=FAKE, o_dtype=0,
                final_state=FAKE, workspace=FAKE, workspace_bytes=1 << 40, stream=None)
    args.update(over)
    return kda.library().kda_chunk_prefill(
        args["q"], args["k"], args["v"], args["z"], args["A"], args["b"], args["initial_state"], args["cu"],
        args["cu_host"], args["batch"], args["seq_len"], args["num_seqs"], args["num_heads"], args["d_k"],
        args["d_v"], args["o"], args["o_dtype"], args["final_state"], args["workspace"], args["workspace_bytes"],
        args["stream"])


def _host_cu(vals):
    arr = (ctypes.c_int32 * len(vals))(*vals)
    return ctypes.cast(arr, ctypes.c_void_p), arr


@pytest.mark.parametrize("over,code", [
    (dict(d_k=64), KDA_ERR_UNSUPPORTED),
    (dict(d_v=256), KDA_ERR_UNSUPPORTED),
    (dict(o_dtype=7), KDA_ERR_UNSUPPORTED),
    (dict(num_heads=0), KDA_ERR_SHAPE),
    (dict(seq_len=-1), KDA_ERR_SHAPE),
    (dict(batch=2, num_seqs=1), KDA_ERR_SHAPE),
    (dict(batch=2, num_seqs=2, cu=FAKE), KDA_ERR_SHAPE),
    (dict(seq_len=1 << 31), KDA_ERR_SHAPE),
    (dict(num_heads=65536), KDA_ERR_SHAPE),                       # heads are grid y
    (dict(seq_len=1 << 30, num_heads=4096), KDA_ERR_SHAPE),        # chunk slots x heads >= 2^31
    (dict(q=None), KDA_ERR_NULL),
    (dict(final_state=None), KDA_ERR_NULL),
    (dict(workspace=None), KDA_ERR_NULL),
    (dict(A=None), KDA_ERR_NULL),
    (dict(q=FAKE + 8), KDA_ERR_ALIGN),
    (dict(z=FAKE + 4), KDA_ERR_ALIGN),
    (dict(initial_state=FAKE + 8), KDA_ERR_ALIGN),
    (dict(workspace=FAKE + 16), KDA_ERR_ALIGN),
    (dict(workspace_bytes=1024), KDA_ERR_WORKSPACE),
])
def test_prefill_argument_checks(over, code):
    assert _prefill(**over) == code


def _prefill_noalloc(**over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, A=FAKE, b=FAKE, initial_state=None, cu=None, cu_host=None,
                batch=1, seq_len=256, num_seqs=1, num_heads=2, d_k=128, d_v=128, o=FAKE, o_dtype=0,
                final_state=FAKE, stream=None)
    args.update(over)
    fn = kda.library().kda_chunk_prefill_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp, vp]
    fn.restype = ctypes.c_int
    return fn(args["q"], args["k"], args["v"], args["z"], args["A"], args["b"], args["initial_state"], args["cu"],
              args["cu_host"], args["batch"], args["seq_len"], args["num_seqs"], args["num_heads"], args["d_k"],
              args["d_v"], args["o"], args["o_dtype"], args["final_state"], args["stream"])


@pytest.mark.parametrize("over", [
    dict(d_k=64), dict(o_dtype=7), dict(num_heads=0), dict(seq_len=-1), dict(batch=2, num_seqs=1),
    dict(batch=2, num_seqs=2, cu=FAKE), dict(seq_len=1 << 31), dict(batch=2, seq_len=1 << 40),
    dict(num_heads=65536), dict(seq_len=1 << 30, num_heads=4096), dict(q=None), dict(final_state=None),
    dict(A=None), dict(q=FAKE + 8), dict(initial_state=FAKE + 8),
    # the same bad sizes on a batch too large for the fixed scratch: the argument error wins
    dict(d_k=64, seq_len=1 << 20, num_heads=12), dict(num_heads=70000, seq_len=1 << 20),
    dict(batch=3, num_seqs=3, cu=FAKE, seq_len=1 << 20, num_heads=12),
])
def test_noalloc_argument_checks_match_the_workspace_entry_point(over):
    """The entry point without a workspace checks its arguments exactly as
    kda_chunk_prefill does and returns the same codes; none of these calls reaches the
    scratch lookup or a launch."""
    expect = _prefill(**over)
    assert expect not in (KDA_OK, KDA_ERR_WORKSPACE)
    assert _prefill_noalloc(**over) == expect


def test_noalloc_refuses_a_batch_larger_than_its_scratch_on_the_host():
    assert _prefill_noalloc(seq_len=1 << 20, num_heads=12) == KDA_ERR_WORKSPACE
    ptr, keep = _host_cu([0, 100, 90, 256])
    assert _prefill_noalloc(cu=FAKE, cu_host=ptr, num_seqs=3) == KDA_ERR_SEQLENS


def test_prefill_host_cu_seqlens_checks():
    for vals, code in (([0, 100, 90, 256], KDA_ERR_SEQLENS),   # falls
                       ([1, 100, 200, 256], KDA_ERR_SEQLENS),  # does not start at 0
                       ([0, 100, 200, 255], KDA_ERR_SEQLENS)): # does not end at the token count
        ptr, keep = _host_cu(vals)
        assert _prefill(cu=FAKE, cu_host=ptr, num_seqs=3) == code


def test_prefill_empty_batch_is_ok():
    assert _prefill(batch=0, num_seqs=0, q=None, k=None, v=None, z=None, b=None, o=None) == KDA_OK


def _decode(**over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, A=FAKE, b=FAKE, state=FAKE, o=FAKE, num_seqs=4, num_heads=2,
                d_k=128, d_v=128, stream=None)
    args.update(over)
    return kda.library().kda_recurrent_decode(
        args["q"], args["k"], args["v"], args["z"], args["A"], args["b"], args["state"], args["o"],
        args["num_seqs"], args["num_heads"], args["d_k"], args["d_v"], args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(d_k=96), KDA_ERR_UNSUPPORTED),
    (dict(num_heads=0), KDA_ERR_SHAPE),
    (dict(num_seqs=-3), KDA_ERR_SHAPE),
    (dict(num_seqs=1 << 30, num_heads=4), KDA_ERR_SHAPE),          # pairs >= 2^31
    (dict(num_seqs=1, num_heads=65536), KDA_ERR_SHAPE),
    (dict(state=None), KDA_ERR_NULL),
    (dict(o=None), KDA_ERR_NULL),
    (dict(v=FAKE + 2), KDA_ERR_ALIGN),
    (dict(state=FAKE + 8), KDA_ERR_ALIGN),
    (dict(num_seqs=0), KDA_OK),
])
def test_decode_argument_checks(over, code):
    assert _decode(**over) == code


def _verify(**over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, z=FAKE, A=FAKE, b=FAKE, state=FAKE, state_out=None, o=FAKE, gk=FAKE,
                beta=FAKE, num_seqs=4, num_heads=2, m=8, d_k=128, d_v=128, stream=None)
    args.update(over)
    return kda.library().kda_recurrent_verify(
        args["q"], args["k"], args["v"], args["z"], args["A"], args["b"], args["state"], args["state_out"],
        args["o"], args["gk"], args["beta"], args["num_seqs"], args["num_heads"], args["m"], args["d_k"],
        args["d_v"], args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(d_v=64), KDA_ERR_UNSUPPORTED),
    (dict(m=17), KDA_ERR_UNSUPPORTED),
    (dict(m=-1), KDA_ERR_SHAPE),
    (dict(num_seqs=1 << 30, num_heads=4), KDA_ERR_SHAPE),
    (dict(num_heads=0), KDA_ERR_SHAPE),
    (dict(state=None), KDA_ERR_NULL),
    (dict(z=None), KDA_ERR_NULL),
    (dict(o=FAKE + 4), KDA_ERR_ALIGN),
    (dict(gk=FAKE + 8), KDA_ERR_ALIGN),
    (dict(state_out=FAKE + 8), KDA_ERR_ALIGN),
    (dict(m=0), KDA_OK),
    (dict(num_seqs=0), KDA_OK),
])
def test_verify_argument_checks(over, code):
    assert _verify(**over) == code


def _fold(**over):
    args = dict(k=FAKE, v=FAKE, gk=FAKE, beta=FAKE, acc=FAKE, state=FAKE, num_seqs=4, num_heads=2, m=8,
                d_k=128, d_v=128, stream=None)
    args.update(over)
    return kda.library().kda_replay_fold(
        args["k"], args["v"], args["gk"], args["beta"], args["acc"], args["state"], args["num_seqs"],
        args["num_heads"], args["m"], args["d_k"], args["d_v"], args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(d_k=256), KDA_ERR_UNSUPPORTED),
    (dict(m=KDA_MAX_REPLAY + 1), KDA_ERR_UNSUPPORTED),
    (dict(num_seqs=-1), KDA_ERR_SHAPE),
    (dict(num_seqs=1 << 30, num_heads=4), KDA_ERR_SHAPE),
    (dict(acc=None), KDA_ERR_NULL),
    (dict(gk=None), KDA_ERR_NULL),
    (dict(acc=FAKE + 2), KDA_ERR_ALIGN),
    (dict(k=FAKE + 8), KDA_ERR_ALIGN),
    (dict(m=0), KDA_OK),
])
def test_fold_argument_checks(over, code):
    assert _fold(**over) == code


def test_max_replay_constant_matches_header():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    m = re.search(r"#define KDA_MAX_REPLAY_TOKENS (\d+)", text)
    assert m and int(m.group(1)) == KDA_MAX_REPLAY == kda.MAX_REPLAY_TOKENS


def _fused(**over):
    args = dict(xq=FAKE, xk=FAKE, xv=FAKE, cs=FAKE, cw=FAKE, z=FAKE, A=FAKE, b=FAKE, g=FAKE, nw=FAKE, e1=1e-6,
                e2=1e-6, state=FAKE, y=FAKE, num_seqs=4, num_heads=2, d_k=128, d_v=128, stream=None)
    args.update(over)
    return kda.library().kda_fused_decode(
        args["xq"], args["xk"], args["xv"], args["cs"], args["cw"], args["z"], args["A"], args["b"], args["g"],
        args["nw"], args["e1"], args["e2"], args["state"], args["y"], args["num_seqs"], args["num_heads"],
        args["d_k"], args["d_v"], args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(d_k=64), KDA_ERR_UNSUPPORTED),
    (dict(e1=-1.0), KDA_ERR_UNSUPPORTED),
    (dict(e2=float("nan")), KDA_ERR_UNSUPPORTED),
    (dict(num_heads=0), KDA_ERR_SHAPE),
    (dict(num_seqs=1 << 30, num_heads=4), KDA_ERR_SHAPE),
    (dict(cs=None), KDA_ERR_NULL),
    (dict(nw=None), KDA_ERR_NULL),
    (dict(cw=FAKE + 4), KDA_ERR_ALIGN),
    (dict(g=FAKE + 8), KDA_ERR_ALIGN),
    (dict(num_seqs=0), KDA_OK),
])
def test_fused_decode_argument_checks(over, code):
    assert _fused(**over) == code
