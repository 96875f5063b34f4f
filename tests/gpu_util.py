"""Shared helpers of the GPU parity tests: error measures, the stated tolerances,
and oracle runs on a sample of (sequence, head) units of a large batch."""
import numpy as np
import torch

import oracle

# Tolerances of the CUDA path against the fp64 oracle.
PREFILL_O_TOL = 1e-2      # max |o - o_ref| / rms(o_ref), o kept in fp32
PREFILL_S_TOL = 5e-3      # ||S - S_ref||_F / ||S_ref||_F
DECODE_TOL = 1e-4         # max |x - x_ref| / rms(x_ref) for o, Frobenius for S
BF16_HALF_ULP = 2.0 ** -8  # bound on |bf16(x) - x| / |x| of round-to-nearest


def np64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def max_over_rms(x, ref):
    x, ref = np64(x), np64(ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(x - ref))) / max(rms, 1e-300)


def rel_frob(x, ref):
    x, ref = np64(x), np64(ref)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_prefill_close(o, S, o_ref, S_ref, what=""):
    o64 = np64(o)
    if o.dtype == torch.bfloat16:
        # the final rounding to bf16 adds at most half an ulp of each output
        ref = np64(o_ref)
        rms = float(np.sqrt(np.mean(ref ** 2)))
        bound = PREFILL_O_TOL * rms + BF16_HALF_ULP * np.abs(ref)
        excess = float(np.max(np.abs(o64 - ref) - bound))
        assert excess <= 0, "%s bf16 o exceeds tol + rounding by %.3e" % (what, excess)
    else:
        e = max_over_rms(o64, o_ref)
        assert e <= PREFILL_O_TOL, "%s o max/rms %.3e > %.1e" % (what, e, PREFILL_O_TOL)
    if S is not None:
        e = rel_frob(S, S_ref)
        assert e <= PREFILL_S_TOL, "%s S relF %.3e > %.1e" % (what, e, PREFILL_S_TOL)


def oracle_units(inp, cu, units, S0=None, threads=0):
    """Oracle of selected (sequence n, head h) units of a packed batch.

    inp: dict of CPU tensors shaped [1, T_total, H, ...] (or [T_total, H, ...]); cu: list
    of token offsets. Returns {(n, h): (o [len, 128] fp64, S [128, 128] fp64)}.
    """
    out = {}
    def flat(t):
        return t.reshape((-1,) + tuple(t.shape[-2:])) if t.dim() >= 3 else t.reshape(-1, t.shape[-1])
    q, k, v, z = (flat(inp[x]) for x in ("q", "k", "v", "z"))
    b = inp["b"].reshape(-1, inp["b"].shape[-1])
    A = inp["A"]
    for (n, h) in units:
        a, e = int(cu[n]), int(cu[n + 1])
        s0 = None if S0 is None else S0[n:n + 1, h:h + 1]
        o, S = oracle.kda_forward(q[a:e, h:h + 1], k[a:e, h:h + 1], v[a:e, h:h + 1], z[a:e, h:h + 1],
                                  A[h:h + 1], b[a:e, h:h + 1], S0=s0, threads=threads)
        out[(n, h)] = (o[:, 0], S[0, 0])
    return out
