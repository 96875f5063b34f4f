"""Pins of the KDA oracle against what the pages and the mathematics fix.

Each pin takes an oracle handle (oracle.Oracle) and raises AssertionError when the
oracle disagrees with something other than itself: a worked example printed on
the pages (tests/golden), a closed form, an invariant, or a brute-force product of
explicit matrices. tests/test_oracle_pins.py runs them on the real oracle;
tests/test_oracle_mutants.py runs them on deliberately broken copies of it and
checks that every planted mistake trips at least one pin.
"""
import numpy as np

from oracle.chunkwise import chunkwise
from tests.conftest import read_golden

NEG_INF = np.float32(-np.inf)
POS_INF = np.float32(np.inf)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rng_case(seed, T, dk, dv, la_lo=-5.0):
    r = np.random.default_rng(seed)
    q = _unit_rows(r.standard_normal((T, 1, dk)))
    k = _unit_rows(r.standard_normal((T, 1, dk)))
    v = r.standard_normal((T, 1, dv))
    la = r.uniform(la_lo, 0.0, (T, 1, dk))
    beta = r.uniform(0.0, 1.0, (T, 1))
    S0 = r.standard_normal((1, 1, dk, dv))
    return q, k, v, la, beta, S0


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b)))) if b.size else 1.0
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol * scale, "%s: max |diff| %.3e > %.1e (scale %.3g)" % (what, err, tol, scale)


# --- worked examples printed on the pages ------------------------------------------


def pin_linear_attention_worked_example(orc):
    """Blog §3: d=1, (k,v) = (2,5), (3,7), q3 = 4 -> S2 = 31, o3 = 124 (no decay, no delta, unit write)."""
    g = read_golden("linear_attention_d1.txt")
    k = np.array([g["k1"], g["k2"], 0.0]).reshape(3, 1, 1)
    v = np.array([g["v1"], g["v2"], 0.0]).reshape(3, 1, 1)
    q = np.array([0.0, 0.0, g["q3"]]).reshape(3, 1, 1)
    la = np.zeros((3, 1, 1))
    beta = np.ones((3, 1))
    o, S = orc.recurrence(q[:2], k[:2], v[:2], la[:2], beta[:2], delta=False)
    _close(S[0, 0, 0, 0], g["S2"], 0, "S2")
    o, S = orc.recurrence(q, k, v, la, beta, delta=False)
    _close(o[2, 0, 0], g["o3"], 0, "o3")
    for C in (1, 2, 3):
        oc, Sc = chunkwise(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], np.zeros((1, 1)), C, delta=False)
        _close(oc[2, 0], g["o3"], 1e-15, "chunkwise o3 C=%d" % C)
        _close(Sc[0, 0], g["S2"], 1e-15, "chunkwise S C=%d" % C)


def pin_deltanet_worked_example(orc):
    """Blog §7.4: DeltaNet, C=2, k=1, v=(5,7), beta=(0.5,0.4): S1=2.5, S2=4.3, u=(2.5,1.8)."""
    g = read_golden("deltanet_chunk_c2.txt")
    k = np.array([g["k1"], g["k2"]]).reshape(2, 1, 1)
    v = np.array([g["v1"], g["v2"]]).reshape(2, 1, 1)
    q = np.ones((2, 1, 1))           # o_t = S_t^T q_t with q = 1 reads S_t
    la = np.zeros((2, 1, 1))
    beta = np.array([g["beta1"], g["beta2"]]).reshape(2, 1)
    o, S = orc.recurrence(q, k, v, la, beta, delta=True)
    _close(o[:, 0, 0], [g["S1"], g["S2"]], 1e-15, "recurrent S1, S2")
    _close(S[0, 0, 0, 0], g["S2"], 1e-15, "final S2")
    oc, Sc, us = chunkwise(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], np.zeros((1, 1)), 2, return_u=True)
    _close(us[0][:, 0], [g["u1"], g["u2"]], 1e-15, "UT solve u")
    _close(Sc[0, 0], g["S2"], 1e-15, "chunkwise S2")
    # the same example through the gate: z = -inf gives a = 1; beta from b = logit(beta)
    z = np.full((2, 1, 1), NEG_INF, dtype=np.float32)
    A = np.zeros(1, dtype=np.float32)
    b = np.log(np.array([g["beta1"], g["beta2"]]) / (1 - np.array([g["beta1"], g["beta2"]])))
    b = b.astype(np.float32).reshape(2, 1)
    o, S = orc.kda_forward(q, k, v, z, A, b)
    _close(o[:, 0, 0], [g["S1"], g["S2"]], 1e-7, "gate path S1, S2")


# --- the gate: closed forms -------------------------------------------------------------


def pin_gate_closed_forms(orc):
    """Blog §5.4: log a = -5*sigmoid(e^A z) in (-5, 0); beta = sigmoid(b) (§5.3)."""
    ln3 = np.log(3.0)
    z = np.array([[[0.0, ln3, -ln3, POS_INF, NEG_INF, 2 * ln3]]], dtype=np.float32)   # [1,1,6]
    b = np.array([[0.0]], dtype=np.float32)
    A = np.zeros(1, dtype=np.float32)
    la, beta = orc.gate(z, A, b)
    la = la[0, 0]
    _close(la[0], -2.5, 0, "sigmoid(0) = 1/2")
    _close(la[1], -3.75, 1e-7, "sigmoid(ln 3) = 3/4")
    _close(la[2], -1.25, 1e-7, "sigmoid(-ln 3) = 1/4")
    assert la[3] == -5.0, "z=+inf must give the lower bound -5 exactly"
    assert la[4] == 0.0, "z=-inf must give a = 1 exactly"
    _close(la[5], -5.0 * 9.0 / 10.0, 1e-7, "sigmoid(ln 9) = 9/10")
    _close(beta[0, 0], 0.5, 0, "beta(0)")
    # e^A multiplies z: A = ln 3 with z = 1 is sigmoid(3) ... compare with A = 0, z = 3
    A2 = np.array([np.log(3.0)], dtype=np.float32)
    z2 = np.array([[[1.0, -2.0]]], dtype=np.float32)
    z3 = np.array([[[3.0, -6.0]]], dtype=np.float32)
    la2, _ = orc.gate(z2, A2, b)
    la3, _ = orc.gate(z3, A, b)
    _close(la2, la3, 1e-6, "e^A scales z")
    # beta closed forms: sigmoid(ln 4) = 4/5, b = +-inf gives exactly 1 and 0
    bb = np.array([[np.log(4.0)], [POS_INF], [NEG_INF]], dtype=np.float32)
    zz = np.zeros((3, 1, 1), dtype=np.float32)
    _, beta = orc.gate(zz, A, bb)
    _close(beta[0, 0], 0.8, 1e-7, "sigmoid(ln 4)")
    assert beta[1, 0] == 1.0 and beta[2, 0] == 0.0, "b = +-inf must give beta = 1, 0 exactly"
    # range and monotonicity over finite inputs
    r = np.random.default_rng(1)
    # |e^A z| stays below ~15 so that fp64 sigmoid is not yet exactly 0 or 1
    zr = np.sort(r.standard_normal(200).astype(np.float32)).reshape(1, 1, 200)
    Ar = np.array([np.log(3.0)], dtype=np.float32)
    la, _ = orc.gate(zr, Ar, b)
    la = la[0, 0]
    assert np.all(la < 0) and np.all(la > -5), "log a must lie in (-5, 0)"
    assert np.all(np.diff(la) <= 0), "log a must fall as z grows"


# --- invariants and closed forms of the recurrence --------------------------------------


def pin_single_token_reads_after_write(orc):
    """o_t = S_t^T q_t after the write: from S0 = 0 one token gives o = beta (q.k) v."""
    q, k, v, la, beta, _ = _rng_case(2, 1, 8, 5)
    o, S = orc.recurrence(q, k, v, la, beta, delta=True)
    expect = beta[0, 0] * float(q[0, 0] @ k[0, 0]) * v[0, 0]
    _close(o[0, 0], expect, 1e-14, "one token from zero state")
    _close(S[0, 0], beta[0, 0] * np.outer(k[0, 0], v[0, 0]), 1e-14, "state after one token")


def pin_retrieval(orc):
    """beta = 1 and |k| = 1: S_t^T k_t = v_t for any decay and any prior state (delta rule)."""
    T, dk, dv = 10, 8, 6
    q, k, v, la, _, S0 = _rng_case(3, T, dk, dv)
    S = S0
    for t in range(T):
        o, S = orc.recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], np.ones((1, 1)), S0=S)
        _close(S[0, 0].T @ k[t, 0], v[t, 0], 1e-12, "retrieval at t=%d" % t)


def pin_identity_when_no_decay_no_write(orc):
    """a = 1 and beta = 0 leave the state unchanged; o_t = S0^T q_t."""
    T, dk, dv = 7, 8, 6
    q, k, v, _, _, S0 = _rng_case(4, T, dk, dv)
    o, S = orc.recurrence(q, k, v, np.zeros((T, 1, dk)), np.zeros((T, 1)), S0=S0)
    assert np.array_equal(S, S0), "state must not change"
    _close(o[:, 0], q[:, 0] @ S0[0, 0], 1e-13, "o = S0^T q")


def pin_scalar_decay_closed_form(orc):
    """Scalar decay (RetNet row of the variant table, blog §4) with beta = 0: S_T = (prod a) S0."""
    T, dk, dv = 9, 8, 6
    q, k, v, _, _, S0 = _rng_case(5, T, dk, dv)
    r = np.random.default_rng(6)
    la_t = r.uniform(-5, 0, T)
    la = np.repeat(la_t[:, None, None], dk, axis=2)
    o, S = orc.recurrence(q, k, v, la, np.zeros((T, 1)), S0=S0)
    _close(S[0, 0], np.exp(la_t.sum()) * S0[0, 0], 1e-13, "scalar decay")


def pin_gla_closed_form(orc):
    """Per-channel decay without the delta term (GLA row, blog §4, unrolled as in §7.2):
    S_t = Diag(g_t) S0 + sum_{j<=t} Diag(g_t/g_j) beta_j k_j v_j^T, o_t = S_t^T q_t."""
    T, dk, dv = 8, 6, 5
    q, k, v, la, beta, S0 = _rng_case(7, T, dk, dv)
    o, S = orc.recurrence(q, k, v, la, beta, S0=S0, delta=False)
    G = np.cumsum(la[:, 0], axis=0)
    for t in range(T):
        St = np.exp(G[t])[:, None] * S0[0, 0]
        for j in range(t + 1):
            St = St + (np.exp(G[t] - G[j]) * beta[j, 0] * k[j, 0])[:, None] * v[j, 0][None, :]
        _close(o[t, 0], St.T @ q[t, 0], 1e-12, "GLA o at t=%d" % t)
    _close(S[0, 0], St, 1e-12, "GLA final state")


def pin_orthonormal_keys(orc):
    """a = 1 and orthonormal keys e_{p(t)}: each token rewrites only its own row,
    S_T[p(t)] = S0[p(t)] + beta_t (v_t - S0[p(t)]) (no interference, blog §5.1)."""
    dk, dv = 8, 5
    perm = [5, 2, 7, 0, 3]
    T = len(perm)
    r = np.random.default_rng(8)
    k = np.zeros((T, 1, dk))
    for t, p in enumerate(perm):
        k[t, 0, p] = 1.0
    q = _unit_rows(r.standard_normal((T, 1, dk)))
    v = r.standard_normal((T, 1, dv))
    beta = r.uniform(0, 1, (T, 1))
    S0 = r.standard_normal((1, 1, dk, dv))
    o, S = orc.recurrence(q, k, v, np.zeros((T, 1, dk)), beta, S0=S0)
    expect = S0[0, 0].copy()
    for t, p in enumerate(perm):
        expect[p] = S0[0, 0, p] + beta[t, 0] * (v[t, 0] - S0[0, 0, p])
    _close(S[0, 0], expect, 1e-14, "orthonormal keys")


def pin_brute_force_products(orc):
    """Tiny cases against explicit d x d matrices: with A_m = (I - beta_m k_m k_m^T) Diag(a_m)
    (blog §5.2), S_t = (A_t ... A_1) S0 + sum_j (A_t ... A_{j+1}) beta_j k_j v_j^T."""
    for seed, (T, d) in enumerate([(1, 1), (5, 1), (6, 2), (8, 4), (7, 3)]):
        q, k, v, la, beta, S0 = _rng_case(20 + seed, T, d, d)
        o, S = orc.recurrence(q, k, v, la, beta, S0=S0)
        mats = [(np.eye(d) - beta[m, 0] * np.outer(k[m, 0], k[m, 0])) @ np.diag(np.exp(la[m, 0]))
                for m in range(T)]
        for t in range(T):
            P = np.eye(d)
            for m in range(t, -1, -1):
                P = P @ mats[m]
            St = P @ S0[0, 0]
            for j in range(t + 1):
                Pj = np.eye(d)
                for m in range(t, j, -1):
                    Pj = Pj @ mats[m]
                St = St + Pj @ (beta[j, 0] * np.outer(k[j, 0], v[j, 0]))
            _close(o[t, 0], St.T @ q[t, 0], 1e-12, "brute force o (T=%d d=%d t=%d)" % (T, d, t))
        _close(S[0, 0], St, 1e-12, "brute force S (T=%d d=%d)" % (T, d))


def pin_chunkwise_equals_recurrence(orc):
    """The chunk algebra (blog §7) equals the recurrence for every chunk size, ragged tails
    included, at the decay bound as well as for random decay."""
    for seed, (T, dk, dv, la_lo) in enumerate([(37, 8, 8, -5.0), (100, 16, 8, -5.0), (64, 8, 4, -0.5)]):
        q, k, v, la, beta, S0 = _rng_case(40 + seed, T, dk, dv, la_lo)
        o, S = orc.recurrence(q, k, v, la, beta, S0=S0)
        for C in (1, 2, 3, 8, 16, 64, T):
            oc, Sc = chunkwise(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], S0[0, 0], C)
            _close(oc, o[:, 0], 1e-12, "chunkwise o (T=%d C=%d)" % (T, C))
            _close(Sc, S[0, 0], 1e-12, "chunkwise S (T=%d C=%d)" % (T, C))
    # every token at the lower bound log a = -5: exp(G_i - G_j) spans e^-320 inside a chunk
    q, k, v, _, beta, S0 = _rng_case(50, 70, 8, 8)
    la = np.full((70, 1, 8), -5.0)
    o, S = orc.recurrence(q, k, v, la, beta, S0=S0)
    oc, Sc = chunkwise(q[:, 0], k[:, 0], v[:, 0], la[:, 0], beta[:, 0], S0[0, 0], 64)
    _close(oc, o[:, 0], 1e-12, "chunkwise o at the bound")
    _close(Sc, S[0, 0], 1e-12, "chunkwise S at the bound")


def pin_packing_and_splits(orc):
    """Sequences are independent: packed varlen equals separate runs, an empty sequence
    returns its initial state, and the split into threads and column blocks changes nothing."""
    dk, dv, H = 8, 6, 2
    lens = [5, 0, 12, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    r = np.random.default_rng(60)
    q = _unit_rows(r.standard_normal((T, H, dk)))
    k = _unit_rows(r.standard_normal((T, H, dk)))
    v = r.standard_normal((T, H, dv))
    la = r.uniform(-5, 0, (T, H, dk))
    beta = r.uniform(0, 1, (T, H))
    S0 = r.standard_normal((len(lens), H, dk, dv))
    o, S = orc.recurrence(q, k, v, la, beta, S0=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        if e == a:
            assert np.array_equal(S[n], S0[n]), "empty sequence must return its initial state"
            continue
        on, Sn = orc.recurrence(q[a:e], k[a:e], v[a:e], la[a:e], beta[a:e], S0=S0[n:n + 1])
        assert np.array_equal(on, o[a:e]) and np.array_equal(Sn[0], S[n]), "packing changed sequence %d" % n
    for threads, cb in ((1, 1), (3, 4), (0, dv)):
        o2, S2 = orc.recurrence(q, k, v, la, beta, S0=S0, cu_seqlens=cu, threads=threads, col_block=cb)
        assert np.array_equal(o2, o) and np.array_equal(S2, S), "thread/column split changed the result"
    # heads are independent: permuting them permutes the outputs
    perm = [1, 0]
    o3, S3 = orc.recurrence(q[:, perm], k[:, perm], v[:, perm], la[:, perm], beta[:, perm],
                            S0=S0[:, perm], cu_seqlens=cu)
    assert np.array_equal(o3, o[:, perm]) and np.array_equal(S3, S[:, perm]), "head permutation"


def pin_prefill_then_decode(orc):
    """Running T tokens then m more from the returned state equals running T + m at once
    ('Kimi K3', llm.rainlin.net: the chunk and recurrent paths must agree on the state)."""
    T, m, dk, dv = 20, 4, 8, 8
    q, k, v, la, beta, S0 = _rng_case(70, T + m, dk, dv)
    o, S = orc.recurrence(q, k, v, la, beta, S0=S0)
    o1, S1 = orc.recurrence(q[:T], k[:T], v[:T], la[:T], beta[:T], S0=S0)
    outs = [o1]
    for t in range(T, T + m):
        ot, S1 = orc.recurrence(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], beta[t:t + 1], S0=S1)
        outs.append(ot)
    assert np.array_equal(np.concatenate(outs), o) and np.array_equal(S1, S), "split run differs"


def pin_replay_fold_matches_snapshots(orc):
    """ReplaySSM ('Kimi K3 attention deep dive', §6.2): replaying the accepted prefix of a
    draft window from the checkpoint gives the state that a snapshot taken after that many
    single-token steps holds, for every accepted count (clamped to the window)."""
    import oracle as oracle_mod
    N, H, m, dk, dv = 3, 2, 5, 8, 8
    rng = np.random.default_rng(91)
    q = _unit_rows(rng.standard_normal((N * m, H, dk)))
    k = _unit_rows(rng.standard_normal((N * m, H, dk)))
    v = rng.standard_normal((N * m, H, dv))
    z = rng.standard_normal((N * m, H, dk)).astype(np.float32)
    A = np.log(rng.uniform(1, 16, H)).astype(np.float32)
    b = rng.standard_normal((N * m, H)).astype(np.float32)
    S0 = 0.1 * rng.standard_normal((N, H, dk, dv))
    o, S_all, la, beta = oracle_mod.verify(q, k, v, z, A, b, S0, m)
    # snapshots: one token at a time per sequence
    snaps = np.empty((m + 1, N, H, dk, dv))
    snaps[0] = S0
    for n in range(N):
        S = S0[n:n + 1]
        for t in range(m):
            r = slice(n * m + t, n * m + t + 1)
            ot, S = orc.recurrence(q[r], k[r], v[r], la[r], beta[r], S0=S)
            assert np.array_equal(ot, o[r]), "verify output differs from the single-token step"
            snaps[t + 1, n] = S[0]
    assert np.array_equal(snaps[m], S_all), "verify end state"
    for accepted in ([0, 0, 0], [1, 2, 3], [5, 0, 4], [m + 3, -2, 2]):
        S = oracle_mod.replay_fold(k, v, la, beta, S0, accepted, m)
        for n in range(N):
            a = min(max(accepted[n], 0), m)
            assert np.array_equal(S[n], snaps[a, n]), "fold of %d tokens (seq %d)" % (a, n)


def pin_layer_short_conv_matches_numpy_convolve(orc):
    """ShortConv ('Kimi K3 attention deep dive', §2.3: depthwise causal convolution, kernel
    size 4) streamed in pieces with its state equals np.convolve over the whole sequence,
    and its impulse response reads back the taps, newest input on the last tap."""
    from oracle import layer
    rng = np.random.default_rng(101)
    T, C = 13, 5
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, 4))
    ys, st = [], np.zeros((3, C))
    for piece in (slice(0, 1), slice(1, 5), slice(5, 13)):
        y, st = layer.short_conv(x[piece], w, st)
        ys.append(y)
    y = np.concatenate(ys)
    for c in range(C):
        ref = np.convolve(x[:, c], w[c, ::-1])[:T]
        _close(y[:, c], ref, 1e-13, "conv channel %d" % c)
    assert np.array_equal(st, x[T - 3:]), "conv state must hold the last three inputs"
    imp = np.zeros((4, C))
    imp[0] = 1.0
    y, _ = layer.short_conv(imp, w, np.zeros((3, C)))
    for t in range(4):
        assert np.array_equal(y[t], w[:, 3 - t]), "impulse response at %d" % t


def pin_layer_activation_closed_forms(orc):
    """Swish(x) = x sigmoid(x), L2Norm and the gated per-head RMSNorm (same page, §2.3):
    closed forms."""
    from oracle import layer
    assert layer.swish(np.array([0.0]))[0] == 0.0
    _close(layer.swish(np.array([np.log(3.0)])), [0.75 * np.log(3.0)], 1e-15, "swish(ln 3)")
    x = np.linspace(-4, 4, 17)
    _close(layer.swish(x) - layer.swish(-x), x, 1e-14, "swish odd part")
    _close(layer.l2norm(np.array([3.0, 4.0]), 0.0), [0.6, 0.8], 1e-15, "l2norm (3, 4)")
    r = np.random.default_rng(5).standard_normal((4, 9))
    _close(np.linalg.norm(layer.l2norm(r, 0.0), axis=-1), np.ones(4), 1e-14, "unit rows")
    s = np.sum(r[0] ** 2)
    _close(np.sum(layer.l2norm(r[0], 0.5) ** 2), [s / (s + 0.5)], 1e-14, "l2norm epsilon")
    o = np.array([2.0, -2.0, 2.0, -2.0])
    w = np.array([1.0, 2.0, 3.0, 4.0])
    _close(layer.gated_rmsnorm(o, w, np.full(4, np.log(3.0)), 0.0), [0.75, -1.5, 2.25, -3.0], 1e-15,
           "gated rmsnorm")
    _close(layer.gated_rmsnorm(7.0 * r, np.ones(9), np.zeros(9), 0.0),
           0.5 * r / np.sqrt(np.mean(r ** 2, axis=-1, keepdims=True)), 1e-14, "scale invariance, half gate")


def pin_layer_streamed_decode_equals_whole_sequence(orc):
    """Fused decode over T tokens, carrying the recurrent and the conv state, equals the
    whole-sequence form: np.convolve of each channel, Swish, L2Norm, the recurrence over
    all T tokens, then the gated RMSNorm of every output ('Kimi K3', llm.rainlin.net:
    the chunk and recurrent paths must agree, conv state included)."""
    import oracle as oracle_mod
    from oracle import layer
    rng = np.random.default_rng(102)
    N, H, D, T = 2, 2, 8, 6
    X = [rng.standard_normal((N, T, H, D)) for _ in range(3)]
    cw = rng.standard_normal((3, H, D, 4)) * 0.5
    z = rng.standard_normal((N, T, H, D)).astype(np.float32)
    A = np.log(rng.uniform(1, 16, H)).astype(np.float32)
    b = rng.standard_normal((N, T, H)).astype(np.float32)
    g = rng.standard_normal((N, T, H, D))
    nw = 1.0 + 0.1 * rng.standard_normal(D)
    S0 = 0.1 * rng.standard_normal((N, H, D, D))
    eps1, eps2 = 1e-6, 1e-5
    # streamed
    S, cs, ys = S0.copy(), np.zeros((N, 3, 3, H, D)), []
    for t in range(T):
        y, S, cs = layer.fused_decode(X[0][:, t], X[1][:, t], X[2][:, t], cs, cw, z[:, t], A, b[:, t], g[:, t], nw,
                                      S, eps1, eps2)
        ys.append(y)
    # whole sequence
    act = []
    for s in range(3):
        a = np.empty((N, T, H, D))
        for n in range(N):
            for h in range(H):
                for c in range(D):
                    a[n, :, h, c] = np.convolve(X[s][n, :, h, c], cw[s, h, c, ::-1])[:T]
        act.append(layer.swish(a))
    q, k, v = layer.l2norm(act[0], eps1), layer.l2norm(act[1], eps1), act[2]
    la, beta = oracle_mod.gate(z, A, b)
    o, S_ref = orc.recurrence(q, k, v, la, beta, S0=S0)
    y_ref = layer.gated_rmsnorm(o, nw, g, eps2)
    _close(np.stack(ys, axis=1), y_ref, 1e-12, "fused decode outputs")
    _close(S, S_ref, 1e-12, "fused decode state")
    for s in range(3):
        assert np.array_equal(cs[:, s], X[s][:, T - 3:]), "conv state stream %d" % s


ALL_PINS = [
    pin_linear_attention_worked_example,
    pin_deltanet_worked_example,
    pin_gate_closed_forms,
    pin_single_token_reads_after_write,
    pin_retrieval,
    pin_identity_when_no_decay_no_write,
    pin_scalar_decay_closed_form,
    pin_gla_closed_form,
    pin_orthonormal_keys,
    pin_brute_force_products,
    pin_chunkwise_equals_recurrence,
    pin_packing_and_splits,
    pin_prefill_then_decode,
    pin_replay_fold_matches_snapshots,
    pin_layer_short_conv_matches_numpy_convolve,
    pin_layer_activation_closed_forms,
    pin_layer_streamed_decode_equals_whole_sequence,
]
