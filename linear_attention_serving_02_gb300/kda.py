"""Python binding of the KDA C ABI (include/kda.h): argument marshalling only.

Each function here has the name of the C entry point it calls. Tensors are torch
CUDA tensors; the binding checks dtypes and shapes, passes raw pointers, sizes and the
current CUDA stream, and raises KdaError on a non-zero status. Every step of the
computation runs in the CUDA library; if the library cannot be built or loaded the
import fails loudly. There is no other code path.
"""
import ctypes

import torch

from . import build as _build

D = 128
KDA_OUT_BF16 = 0
KDA_OUT_F32 = 1

_LIB = None


class KdaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, status_string(status), status))


def library():
    """The loaded CUDA library (built in-tree on first use if missing or stale)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        lib.kda_version.restype = ctypes.c_int
        lib.kda_chunk_prefill_workspace_size.argtypes = [i64, i32, i32]
        lib.kda_chunk_prefill_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_prefill_launch_count.argtypes = [i64, i32, i32]
        lib.kda_chunk_prefill_launch_count.restype = i32
        lib.kda_chunk_prefill_walk_form.argtypes = [i64, i32, i32]
        lib.kda_chunk_prefill_walk_form.restype = i32
        lib.kda_chunk_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          i32, i64, i32, i32, i32, i32,
                                          vp, i32, vp, vp, ctypes.c_size_t, vp]
        lib.kda_chunk_prefill.restype = ctypes.c_int
        lib.kda_workspace_status.argtypes = [vp, vp]
        lib.kda_workspace_status.restype = ctypes.c_int
        lib.kda_debug_walk_fault.argtypes = [i32, ctypes.c_uint64]
        lib.kda_debug_walk_fault.restype = ctypes.c_int
        lib.kda_debug_segment_ends.argtypes = [i32]
        lib.kda_debug_segment_ends.restype = ctypes.c_int
        lib.kda_recurrent_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]
        lib.kda_recurrent_decode.restype = ctypes.c_int
        lib.kda_recurrent_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
        lib.kda_recurrent_verify.restype = ctypes.c_int
        lib.kda_replay_fold.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
        lib.kda_replay_fold.restype = ctypes.c_int
        f32 = ctypes.c_float
        lib.kda_fused_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, f32, vp, vp, i32, i32, i32, i32,
                                         vp]
        lib.kda_fused_decode.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def status_string(status):
    return library().kda_status_string(int(status)).decode()


kda_status_string = status_string


def kda_version():
    return library().kda_version()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, cuda=True):
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if cuda and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def kda_chunk_prefill_workspace_size(total_tokens, num_seqs, num_heads):
    return int(library().kda_chunk_prefill_workspace_size(int(total_tokens), int(num_seqs), int(num_heads)))


def kda_chunk_prefill_launch_count(total_tokens, num_seqs, num_heads):
    """Kernels one kda_chunk_prefill call with these sizes launches: 3, or 5 for a
    segmented walk (include/kda.h)."""
    return int(library().kda_chunk_prefill_launch_count(int(total_tokens), int(num_seqs), int(num_heads)))


def kda_chunk_prefill_walk_form(total_tokens, num_seqs, num_heads):
    """How the state walk runs for these sizes: 0 one pass per chain, 1 segments whose
    output walks chain the segment maps, 2 segments chained by a combine kernel."""
    return int(library().kda_chunk_prefill_walk_form(int(total_tokens), int(num_seqs), int(num_heads)))


def _prefill_args(q, k, v, z, A, b, initial_state, cu_seqlens, cu_seqlens_host, o, final_state, o_dtype):
    """Checks and sizes shared by both prefill entry points. Returns (batch, seq_len,
    num_seqs, H, host cu_seqlens or None, o, final_state), allocating o and final_state
    with torch when they are not given."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    _need(z, "z", torch.float32)
    _need(A, "A", torch.float32)
    _need(b, "b", torch.float32)
    if q.dim() < 3 or q.shape[-1] != D or k.shape != q.shape or v.shape != q.shape or z.shape != q.shape:
        raise ValueError("q, k, v and z must share one shape [..., H, 128]")
    H = q.shape[-2]
    if A.numel() != H or b.shape != q.shape[:-1]:
        raise ValueError("A must hold H values and b be shaped like q without its last dimension")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a 1-D tensor of num_seqs + 1 offsets")
        if q.dim() == 4 and q.shape[0] != 1:
            raise ValueError("a packed varlen batch wants q as [T_total, H, 128] or [1, T_total, H, 128]")
        batch, seq_len = 1, q.numel() // (H * D)
        num_seqs = cu_seqlens.numel() - 1
    else:
        if q.dim() != 4:
            raise ValueError("dense batch wants q as [B, T, H, 128]")
        batch, seq_len = q.shape[0], q.shape[1]
        num_seqs = batch
    hc = None
    if cu_seqlens_host is not None:
        if cu_seqlens_host.is_cuda or cu_seqlens_host.dim() != 1 or cu_seqlens_host.numel() != num_seqs + 1:
            raise ValueError("cu_seqlens_host must be a 1-D CPU tensor of num_seqs + 1 entries")
        hc = cu_seqlens_host.to(torch.int32).contiguous()
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32)
        if tuple(initial_state.shape) != (num_seqs, H, D, D):
            raise ValueError("initial_state must be [num_seqs, H, 128, 128]")
    if o is None:
        o = torch.empty(q.shape, dtype=o_dtype, device=q.device)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bf16 or fp32")
    _need(o, "o", o.dtype)
    if o.shape != q.shape:
        raise ValueError("o must be shaped like q")
    if final_state is None:
        final_state = torch.empty((num_seqs, H, D, D), dtype=torch.float32, device=q.device)
    _need(final_state, "final_state", torch.float32)
    if tuple(final_state.shape) != (num_seqs, H, D, D):
        raise ValueError("final_state must be [num_seqs, H, 128, 128]")
    return batch, seq_len, num_seqs, H, hc, o, final_state


def kda_chunk_prefill(q, k, v, z, A, b, initial_state=None, cu_seqlens=None, cu_seqlens_host=None,
                      o=None, final_state=None, workspace=None, o_dtype=torch.bfloat16, stream=None):
    """Chunkwise KDA prefill. Returns (o, final_state).

    q, k, v: bf16 [B, T, H, 128] (dense batch) or [T_total, H, 128] with cu_seqlens;
    z: fp32 like q; A: fp32 [H]; b: fp32 [..., H]; initial_state: fp32 [N, H, 128, 128]
    or None; cu_seqlens: int32 CUDA [N+1] or None; cu_seqlens_host: optional CPU int32
    copy of it (validated on the host). o / final_state / workspace are allocated with
    torch when not given.
    """
    batch, seq_len, num_seqs, H, hc, o, final_state = _prefill_args(
        q, k, v, z, A, b, initial_state, cu_seqlens, cu_seqlens_host, o, final_state, o_dtype)
    total = batch * seq_len
    need = kda_chunk_prefill_workspace_size(total, num_seqs, H)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    rc = library().kda_chunk_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(b), _ptr(initial_state), _ptr(cu_seqlens),
        _ptr(hc),
        batch, seq_len, num_seqs, H, D, D,
        _ptr(o), KDA_OUT_F32 if o.dtype == torch.float32 else KDA_OUT_BF16, _ptr(final_state),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != 0:
        raise KdaError("kda_chunk_prefill", rc)
    return o, final_state


def kda_workspace_status(workspace, stream=None):
    """Device-side status of the last prefill that used this workspace (synchronises)."""
    return int(library().kda_workspace_status(_ptr(workspace), _stream(stream)))


def kda_recurrent_decode(q, k, v, z, A, b, state, o=None, stream=None):
    """One decode token per sequence; state [N, H, 128, 128] fp32 is updated in place. Returns o (fp32)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    _need(z, "z", torch.float32)
    _need(A, "A", torch.float32)
    _need(b, "b", torch.float32)
    _need(state, "state", torch.float32)
    N, H = q.shape[0], q.shape[1]
    if o is None:
        o = torch.empty((N, H, D), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32)
    rc = library().kda_recurrent_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(b), _ptr(state), _ptr(o),
                                        N, H, D, D, _stream(stream))
    if rc != 0:
        raise KdaError("kda_recurrent_decode", rc)
    return o


MAX_REPLAY_TOKENS = 16  # KDA_MAX_REPLAY_TOKENS


def kda_recurrent_verify(q, k, v, z, A, b, state, num_tokens, o=None, state_out=None, gk_log=None, beta_log=None,
                         log=True, stream=None):
    """num_tokens draft tokens per sequence from the checkpoint `state` (read only).

    q, k, v: bf16 [N * m, H, 128] token-major (token t of sequence n at row n * m + t);
    z fp32 like q; b fp32 [N * m, H]; state fp32 [N, H, 128, 128]. With log=True the
    gate values are logged (allocated here unless given). state_out (may be `state`)
    receives the state after all m tokens. Returns (o, gk_log, beta_log); o is fp32
    [N * m, H, 128].
    """
    m = int(num_tokens)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    _need(z, "z", torch.float32)
    _need(A, "A", torch.float32)
    _need(b, "b", torch.float32)
    _need(state, "state", torch.float32)
    N, H = state.shape[0], state.shape[1]
    if q.shape[0] != N * m:
        raise ValueError("q has %d rows, expected num_seqs * num_tokens = %d" % (q.shape[0], N * m))
    if o is None:
        o = torch.empty((N * m, H, D), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32)
    if log and gk_log is None:
        gk_log = torch.empty((N * m, H, D), dtype=torch.float32, device=q.device)
    if log and beta_log is None:
        beta_log = torch.empty((N * m, H), dtype=torch.float32, device=q.device)
    for name, t in (("gk_log", gk_log), ("beta_log", beta_log), ("state_out", state_out)):
        if t is not None:
            _need(t, name, torch.float32)
    rc = library().kda_recurrent_verify(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(b), _ptr(state),
                                        _ptr(state_out), _ptr(o), _ptr(gk_log), _ptr(beta_log), N, H, m, D, D,
                                        _stream(stream))
    if rc != 0:
        raise KdaError("kda_recurrent_verify", rc)
    return o, gk_log, beta_log


def kda_replay_fold(k, v, gk_log, beta_log, num_accepted, state, num_tokens, stream=None):
    """Replay the first num_accepted[n] logged tokens of each sequence on `state` in place."""
    m = int(num_tokens)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16)
    _need(gk_log, "gk_log", torch.float32)
    _need(beta_log, "beta_log", torch.float32)
    _need(num_accepted, "num_accepted", torch.int32)
    _need(state, "state", torch.float32)
    N, H = state.shape[0], state.shape[1]
    rc = library().kda_replay_fold(_ptr(k), _ptr(v), _ptr(gk_log), _ptr(beta_log), _ptr(num_accepted), _ptr(state),
                                   N, H, m, D, D, _stream(stream))
    if rc != 0:
        raise KdaError("kda_replay_fold", rc)
    return state


def kda_fused_decode(x_q, x_k, x_v, conv_state, conv_w, z, A, b, g, norm_w, state, y=None, eps_l2=1e-6,
                     eps_rms=1e-6, stream=None):
    """Fused decode layer step (conv -> recurrent update -> gated RMSNorm) for one token per
    sequence. conv_state bf16 [N, 3, 3, H, 128] and state fp32 [N, H, 128, 128] are updated
    in place. Returns y fp32 [N, H, 128]."""
    for name, t in (("x_q", x_q), ("x_k", x_k), ("x_v", x_v), ("conv_state", conv_state)):
        _need(t, name, torch.bfloat16)
    for name, t in (("conv_w", conv_w), ("z", z), ("A", A), ("b", b), ("g", g), ("norm_w", norm_w),
                    ("state", state)):
        _need(t, name, torch.float32)
    N, H = x_q.shape[0], x_q.shape[1]
    if y is None:
        y = torch.empty((N, H, D), dtype=torch.float32, device=x_q.device)
    _need(y, "y", torch.float32)
    rc = library().kda_fused_decode(_ptr(x_q), _ptr(x_k), _ptr(x_v), _ptr(conv_state), _ptr(conv_w), _ptr(z),
                                    _ptr(A), _ptr(b), _ptr(g), _ptr(norm_w), float(eps_l2), float(eps_rms),
                                    _ptr(state), _ptr(y), N, H, D, D, _stream(stream))
    if rc != 0:
        raise KdaError("kda_fused_decode", rc)
    return y


def kda_chunk_prefill_noalloc(q, k, v, z, A, b, initial_state=None, cu_seqlens=None, cu_seqlens_host=None,
                              o=None, final_state=None, o_dtype=torch.bfloat16, stream=None):
    """kda_chunk_prefill on the library's built-in scratch instead of a caller workspace,
    for callers that may not allocate device memory. Same arguments and results as
    kda_chunk_prefill without `workspace` (o and final_state are still allocated here when
    not given; pass them to allocate nothing). Batches larger than the built-in scratch
    raise KdaError with status KDA_ERR_WORKSPACE."""
    lib = library()
    fn = lib.kda_chunk_prefill_noalloc
    if fn.restype is not ctypes.c_int:
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, vp, i32, vp, vp]
        fn.restype = ctypes.c_int
    batch, seq_len, num_seqs, H, hc, o, final_state = _prefill_args(
        q, k, v, z, A, b, initial_state, cu_seqlens, cu_seqlens_host, o, final_state, o_dtype)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(A), _ptr(b), _ptr(initial_state), _ptr(cu_seqlens), _ptr(hc),
            batch, seq_len, num_seqs, H, D, D, _ptr(o), KDA_OUT_F32 if o.dtype == torch.float32 else KDA_OUT_BF16,
            _ptr(final_state), _stream(stream))
    if rc != 0:
        raise KdaError("kda_chunk_prefill_noalloc", rc)
    return o, final_state


def kda_debug_segment_ends(end_factor):
    """Test hook of the segmented walk's long end segments (include/kda.h): end_factor > 0
    forces the first and last segment of every long enough sequence to end_factor segment
    lengths in the combine form; 0 restores the choice the sizes make."""
    rc = library().kda_debug_segment_ends(ctypes.c_int32(end_factor))
    if rc != 0:
        raise KdaError("kda_debug_segment_ends", rc)


def kda_debug_walk_fault(skip_commit_chunk, wait_limit_ns):
    """Test hook of the state walk's failure path (include/kda.h): the walks leave out the
    MMA-completion signal of chunk slot skip_commit_chunk (-1: none) and give up a wait after
    wait_limit_ns nanoseconds. Restore with (-1, 2_000_000_000)."""
    rc = library().kda_debug_walk_fault(ctypes.c_int32(skip_commit_chunk), ctypes.c_uint64(wait_limit_ns))
    if rc != 0:
        raise KdaError("kda_debug_walk_fault", rc)
