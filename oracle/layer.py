"""fp64 statement of the layer steps that the fused decode kernel wraps around the KDA
update ('Kimi K3 attention deep dive', forceinjection.github.io, §2.3 and §6.3):

    q = L2Norm(Swish(ShortConv(x_q)))     k = L2Norm(Swish(ShortConv(x_k)))
    v = Swish(ShortConv(x_v))
    o = KDA decode step (gate from z, A, b; the state updated in place)
    y = RMSNorm(o) * w_norm * sigmoid(g)  (per head, then the output gate)

ShortConv is the depthwise causal convolution of kernel size 4 that the page puts
before the normalisation: channel c of the output at token t is
sum_{j=0..3} w[c, j] * x[t - 3 + j, c], with the three inputs before a sequence's first
token taken from the conv state (zeros for a new sequence). The page fixes no epsilon
for either normalisation, so both are arguments.

TEST INFRASTRUCTURE ONLY, like the rest of this package. Pinned by
tests/oracle_pins.py (pin_layer_*): np.convolve on whole sequences, closed forms of
Swish, L2Norm and the gated RMSNorm, and the streamed form against the whole-sequence
form.
"""
import numpy as np

from . import _as_f32, _as_f64, gate, recurrence

CONV_TAPS = 4


def short_conv(x, w, state):
    """Causal depthwise convolution of new inputs x [T, C] with taps w [C, 4] (oldest tap
    first), continuing from state [3, C] (the three previous inputs, oldest first).
    Returns (y [T, C], new_state [3, C])."""
    x = _as_f64(x)
    w = _as_f64(w)
    st = _as_f64(state)
    T = x.shape[0]
    window = np.concatenate([st, x], axis=0)  # [T + 3, C]
    y = np.zeros_like(x)
    for t in range(T):
        for j in range(CONV_TAPS):
            y[t] += w[:, j] * window[t + j]
    return y, window[T:T + CONV_TAPS - 1].copy()


def swish(x):
    x = _as_f64(x)
    return x / (1.0 + np.exp(-x))


def l2norm(x, eps):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    x = _as_f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gated_rmsnorm(o, w, g, eps):
    """o / sqrt(mean(o^2) + eps) * w * sigmoid(g) over the last axis (one head)."""
    o = _as_f64(o)
    g = _as_f64(g)
    r = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return r * _as_f64(w) / (1.0 + np.exp(-g))


def fused_decode(xq, xk, xv, conv_state, conv_w, z, A, b, g, norm_w, S, eps_l2, eps_rms):
    """One fused decode token for every (sequence n, head h).

    xq, xk, xv [N, H, 128] (the projections before the convolution); conv_state
    [N, 3, 3, H, 128] (stream q/k/v, the three previous inputs oldest first); conv_w
    [3, H, 128, 4]; z [N, H, 128], A [H], b [N, H]; g [N, H, 128] (output-gate
    pre-activation); norm_w [128]; S [N, H, 128, 128]. Returns (y [N, H, 128],
    S_new, conv_state_new), fp64.
    """
    xs = [_as_f64(xq), _as_f64(xk), _as_f64(xv)]
    cs = _as_f64(conv_state)
    cw = _as_f64(conv_w)
    N, H, D = xs[0].shape
    new_cs = np.empty_like(cs)
    act = [np.empty((N, H, D)) for _ in range(3)]
    for n in range(N):
        for h in range(H):
            for s in range(3):
                y, st = short_conv(xs[s][n, h][None, :], cw[s, h], cs[n, s, :, h, :])
                act[s][n, h] = swish(y[0])
                new_cs[n, s, :, h, :] = st
    q = l2norm(act[0], eps_l2)
    k = l2norm(act[1], eps_l2)
    v = act[2]
    la, beta = gate(_as_f32(z).reshape(N, 1, H, D), A, _as_f32(b).reshape(N, 1, H))
    o, S_new = recurrence(q.reshape(N, 1, H, D), k.reshape(N, 1, H, D), v.reshape(N, 1, H, D), la, beta, S0=S)
    y = gated_rmsnorm(o[:, 0], norm_w, g, eps_rms)
    return y, S_new, new_cs
