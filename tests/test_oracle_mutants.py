"""Planted mistakes: each mutant is the oracle's C source with one plausible error
(a flipped sign, a transposed index, a step out of order, a wrong constant), built
into a scratch directory. Every mutant must fail at least one pin; a mutant that
passes them all would show a hole in the pins. CPU only; the real oracle is untouched.
"""
import os
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
from tests.oracle_pins import ALL_PINS

DECAY = ("        for (int64_t c = 0; c < dk; ++c)\n"
         "            for (int64_t j = 0; j < w; ++j) S[c * w + j] *= alpha[c];\n")
PREDICT_END = ("                for (int64_t j = 0; j < w; ++j) p[j] += kt[c] * S[c * w + j];\n")
READ = ("        double *ot = J->o + (t * H + h) * dv + j0;\n"
        "        for (int64_t j = 0; j < w; ++j) ot[j] = 0.0;\n"
        "        for (int64_t c = 0; c < dk; ++c)\n"
        "            for (int64_t j = 0; j < w; ++j) ot[j] += qt[c] * S[c * w + j];\n")
WRITE_COMMENT = "        /* S_t = S' + beta_t k_t (v_t - p)^T */\n"


def _swap(old, new):
    def f(src):
        assert src.count(old) == 1, "mutation anchor not found once: %r" % old
        return src.replace(old, new)
    return f


def _decay_after_prediction(src):
    assert src.count(DECAY) == 1 and src.count(PREDICT_END) == 1
    src = src.replace(DECAY, "")
    return src.replace(PREDICT_END, PREDICT_END + DECAY)


def _read_before_write(src):
    assert src.count(READ) == 1 and src.count(WRITE_COMMENT) == 1
    src = src.replace(READ, "")
    return src.replace(WRITE_COMMENT, READ + WRITE_COMMENT)


MUTANTS = {
    "correction_sign": _swap("(vt[j] - p[j]);", "(vt[j] + p[j]);"),
    "decay_on_columns": _swap("S[c * w + j] *= alpha[c];", "S[c * w + j] *= alpha[j];"),
    "readout_with_key": _swap("ot[j] += qt[c] * S[c * w + j];", "ot[j] += kt[c] * S[c * w + j];"),
    "readout_transposed": _swap("ot[j] += qt[c] * S[c * w + j];", "ot[j] += qt[j] * S[c * w + j];"),
    "prediction_with_query": _swap("p[j] += kt[c] * S[c * w + j];", "p[j] += qt[c] * S[c * w + j];"),
    "gate_bound": _swap("#define KDA_ORACLE_G_MIN (-5.0)", "#define KDA_ORACLE_G_MIN (-4.0)"),
    "gate_missing_exp_A": _swap("const double eA = exp((double)A[h]);", "const double eA = (double)A[h];"),
    "sigmoid_flipped": _swap("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "write_without_beta": _swap("+= bt * kt[c] * (vt[j] - p[j]);", "+= kt[c] * (vt[j] - p[j]);"),
    "initial_state_ignored": _swap("S[c * w + j] = J->S0 ? J->S0[((n * H + h) * dk + c) * dv + j0 + j] : 0.0;",
                                   "S[c * w + j] = 0.0;"),
    "decay_after_prediction": _decay_after_prediction,
    "read_before_write": _read_before_write,
}


def _build_mutant(tmp_path, name, mutate):
    src = open(oracle_build.SRC).read()
    path_c = os.path.join(tmp_path, "mutant_%s.c" % name)
    path_so = os.path.join(tmp_path, "libmutant_%s.so" % name)
    with open(path_c, "w") as f:
        f.write(mutate(src))
    subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-D_GNU_SOURCE", path_c, "-o", path_so, "-lm"], check=True)
    return oracle.Oracle(path_so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    orc = _build_mutant(str(tmp_path), name, MUTANTS[name])
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "planted mistake %r passed every pin" % name


# ---- planted mistakes in the layer steps around the fused decode (oracle/layer.py) ----
LAYER_MUTANTS = {
    "conv_taps_reversed": ("y[t] += w[:, j] * window[t + j]", "y[t] += w[:, CONV_TAPS - 1 - j] * window[t + j]"),
    "conv_state_oldest_kept": ("window[T:T + CONV_TAPS - 1]", "window[:CONV_TAPS - 1]"),
    "swish_sign": ("return x / (1.0 + np.exp(-x))", "return x / (1.0 + np.exp(x))"),
    "l2norm_without_sqrt": ("np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)",
                            "(np.sum(x * x, axis=-1, keepdims=True) + eps)"),
    "rmsnorm_sum_not_mean": ("np.mean(o * o, axis=-1, keepdims=True)", "np.sum(o * o, axis=-1, keepdims=True)"),
    "output_gate_ungated": ("/ (1.0 + np.exp(-g))", "* 1.0"),
    "value_normalised": ("v = act[2]", "v = l2norm(act[2], eps_l2)"),
    "query_not_normalised": ("q = l2norm(act[0], eps_l2)", "q = act[0]"),
}


@pytest.mark.parametrize("name", sorted(LAYER_MUTANTS))
def test_layer_mutant_is_caught(monkeypatch, name):
    import importlib.util

    from oracle import layer
    old, new = LAYER_MUTANTS[name]
    src = open(layer.__file__).read()
    assert src.count(old) == 1, "mutation anchor not found once: %r" % old
    spec = importlib.util.spec_from_loader("oracle._layer_mutant", loader=None, origin=layer.__file__)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), layer.__file__, "exec"), mod.__dict__)
    for fn in ("short_conv", "swish", "l2norm", "gated_rmsnorm", "fused_decode"):
        monkeypatch.setattr(layer, fn, getattr(mod, fn))
    caught = []
    for pin in ALL_PINS:
        if not pin.__name__.startswith("pin_layer_"):
            continue
        try:
            pin(oracle.default())
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "planted mistake %r passed every layer pin" % name
