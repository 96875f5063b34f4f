"""KDA oracle: fp64 CPU statement of Kimi Delta Attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library does not
import, link or call it; the two share no code.

Functions
---------
gate(z, A, b)
    log-decay and write strength of the bounded gate ('From Linear Attention to
    KDA', blog-3d3.pages.dev/posts/150, §5.4 and §5.3), fp64.
recurrence(q, k, v, la, beta, S0, cu_seqlens, delta=True)
    the token-by-token recurrence (same page §5.2; 'Kimi K3 attention deep dive',
    forceinjection.github.io, §2.1-2.2), fp64, in C (oracle/kda_oracle.c).
kda_forward(q, k, v, z, A, b, S0, cu_seqlens)
    gate + recurrence from the raw inputs, each first converted exactly (bf16 or
    fp32 -> fp64) as the GPU receives them. This is the oracle the CUDA path is
    compared with.
verify(q, k, v, z, A, b, S0, num_tokens) / replay_fold(k, v, la, beta, S0, accepted, num_tokens)
    the speculative-decoding pair of ReplaySSM ('Kimi K3 attention deep dive', §6.2):
    num_tokens draft tokens per sequence from a checkpoint, and the replay of each
    sequence's accepted prefix on that checkpoint from the logged gate values.
chunkwise(...)
    (oracle.chunkwise) the chunk algebra of the blog's §7 in fp64, used to pin the
    chunk decomposition against the recurrence.

Every function here is pinned by tests/test_oracle_pins.py against the pages'
worked examples, closed forms and brute force; none is "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

class Oracle:
    """ctypes handle on one build of oracle/kda_oracle.c (the default build, or a
    test's deliberately broken copy)."""

    def __init__(self, lib_path):
        lib = ctypes.CDLL(lib_path)
        d = ctypes.POINTER(ctypes.c_double)
        f = ctypes.POINTER(ctypes.c_float)
        i64 = ctypes.POINTER(ctypes.c_int64)
        lib.kda_oracle_gate.argtypes = [f, f, f, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, d, d]
        lib.kda_oracle_gate.restype = None
        lib.kda_oracle_recurrence.argtypes = [
            ctypes.c_int, d, d, d, d, d, d, i64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            d, d, ctypes.c_int, ctypes.c_int64,
        ]
        lib.kda_oracle_recurrence.restype = ctypes.c_int
        lib.kda_oracle_hardware_threads.argtypes = []
        lib.kda_oracle_hardware_threads.restype = ctypes.c_int
        self.lib = lib

    def gate(self, z, A, b):
        return _gate(self.lib, z, A, b)

    def recurrence(self, q, k, v, la, beta, S0=None, cu_seqlens=None, delta=True, threads=0, col_block=0):
        return _recurrence(self.lib, q, k, v, la, beta, S0, cu_seqlens, delta, threads, col_block)

    def kda_forward(self, q, k, v, z, A, b, S0=None, cu_seqlens=None, threads=0):
        la, beta = self.gate(z, A, b)
        return self.recurrence(q, k, v, la, beta, S0=S0, cu_seqlens=cu_seqlens, delta=True, threads=threads)


_DEFAULT = None


def default():
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(_build.build())
    return _DEFAULT


def _lib():
    return default().lib


def hardware_threads() -> int:
    return int(_lib().kda_oracle_hardware_threads())


def _as_f64(x):
    """Exact conversion to a C-contiguous float64 array (bf16/fp32 -> fp64 is exact)."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu")
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.float()
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _as_f32(x):
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").float().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype != np.float32:
        raise TypeError("gate inputs must be float32 (the precision the kernel receives), got %s" % a.dtype)
    return np.ascontiguousarray(a)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _gate(lib, z, A, b):
    """(la, beta): la = -5*sigmoid(exp(A_h)*z) per channel, beta = sigmoid(b), fp64.

    z: [..., H, dk] fp32; A: [H] fp32; b: [..., H] fp32. Returns la with z's shape and
    beta with b's shape.
    """
    z = _as_f32(z)
    A = _as_f32(A)
    b = _as_f32(b)
    H = A.shape[0]
    dk = z.shape[-1]
    if z.shape[-2] != H or b.shape != z.shape[:-1]:
        raise ValueError("gate: shape mismatch z%s A%s b%s" % (z.shape, A.shape, b.shape))
    T_total = int(np.prod(z.shape[:-2])) if z.ndim > 2 else 1
    la = np.empty(z.shape, dtype=np.float64)
    beta = np.empty(b.shape, dtype=np.float64)
    lib.kda_oracle_gate(_ptr(z, ctypes.c_float), _ptr(A, ctypes.c_float), _ptr(b, ctypes.c_float),
                           T_total, H, dk, _ptr(la, ctypes.c_double), _ptr(beta, ctypes.c_double))
    return la, beta


def _cu(cu_seqlens, n_rows, T):
    """Sequence offsets: given cu_seqlens [N+1], else n_rows sequences of length T each."""
    if cu_seqlens is None:
        return np.arange(n_rows + 1, dtype=np.int64) * T
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    return cu


def _recurrence(lib, q, k, v, la, beta, S0, cu_seqlens, delta, threads, col_block):
    """fp64 recurrence over packed tokens.

    q, k, la: [B, T, H, dk] (or [T_total, H, dk]); v: [..., H, dv]; beta: [..., H];
    S0: [N, H, dk, dv] or None (zeros); cu_seqlens: [N+1] token offsets or None
    (then every one of the B rows is its own sequence). Returns (o [..., H, dv], S [N, H, dk, dv]).
    """
    q = _as_f64(q); k = _as_f64(k); v = _as_f64(v); la = _as_f64(la); beta = _as_f64(beta)
    H, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    if q.ndim == 4:
        B, T = q.shape[0], q.shape[1]
    else:
        B, T = 1, q.shape[0]
    cu = _cu(cu_seqlens, B, T)
    if cu_seqlens is not None and B != 1:
        raise ValueError("cu_seqlens needs B == 1")
    N = cu.shape[0] - 1
    T_total = B * T
    if cu[0] != 0 or cu[-1] != T_total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must rise from 0 to the token count")
    s0 = None
    if S0 is not None:
        s0 = _as_f64(S0)
        if s0.shape != (N, H, dk, dv):
            raise ValueError("S0 must be [N, H, dk, dv]")
    o = np.empty(q.shape[:-1] + (dv,), dtype=np.float64)
    S = np.empty((N, H, dk, dv), dtype=np.float64)
    dp = ctypes.c_double
    rc = lib.kda_oracle_recurrence(
        1 if delta else 0, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(la, dp), _ptr(beta, dp),
        _ptr(s0, dp) if s0 is not None else None, _ptr(cu, ctypes.c_int64),
        N, H, dk, dv, _ptr(o, dp), _ptr(S, dp), int(threads), int(col_block))
    if rc != 0:
        raise RuntimeError("kda_oracle_recurrence failed with %d" % rc)
    return o, S


def gate(z, A, b):
    """(la, beta) of the bounded gate, fp64; see Oracle.gate."""
    return default().gate(z, A, b)


def recurrence(q, k, v, la, beta, S0=None, cu_seqlens=None, delta=True, threads=0, col_block=0):
    """fp64 recurrence over packed tokens; see _recurrence."""
    return default().recurrence(q, k, v, la, beta, S0, cu_seqlens, delta, threads, col_block)


def kda_forward(q, k, v, z, A, b, S0=None, cu_seqlens=None, threads=0):
    """The oracle for the CUDA path: gate then recurrence, fp64, from the exact inputs."""
    return default().kda_forward(q, k, v, z, A, b, S0=S0, cu_seqlens=cu_seqlens, threads=threads)


def verify(q, k, v, z, A, b, S0, num_tokens):
    """Draft window of num_tokens tokens per sequence, read from the checkpoint S0 [N, H, dk, dv].

    Inputs are token-major, token t of sequence n at row n * m + t ([N * m, H, ...]).
    Returns (o, S_after, la, beta) in fp64: every token's output, the state after all m
    tokens, and the logged gate values ('Kimi K3 attention deep dive', §6.2: the verify
    pass stores the gate values its fold will replay).
    """
    m = int(num_tokens)
    N = np.asarray(_as_f64(S0)).shape[0]
    la, beta = gate(z, A, b)
    cu = np.arange(N + 1, dtype=np.int64) * m
    o, S = recurrence(q, k, v, la, beta, S0=S0, cu_seqlens=cu)
    return o, S, la, beta


def replay_fold(k, v, la, beta, S0, accepted, num_tokens):
    """State after each sequence replays the first clamp(accepted[n], 0, m) tokens of its
    window on the checkpoint S0 ('Kimi K3 attention deep dive', §6.2): the recurrence run
    over exactly the accepted prefix, fp64. Returns S [N, H, dk, dv]."""
    m = int(num_tokens)
    k = _as_f64(k); v = _as_f64(v); la = _as_f64(la); beta = _as_f64(beta)
    s0 = _as_f64(S0)
    N = s0.shape[0]
    acc = np.clip(np.asarray(accepted, dtype=np.int64).reshape(N), 0, m)
    rows = np.concatenate([np.arange(n * m, n * m + acc[n], dtype=np.int64) for n in range(N)] +
                          [np.zeros(0, dtype=np.int64)])
    cu = np.concatenate([[0], np.cumsum(acc)]).astype(np.int64)
    q0 = np.zeros_like(k[rows])
    _, S = recurrence(q0, k[rows], v[rows], la[rows], beta[rows], S0=s0, cu_seqlens=cu)
    return S
