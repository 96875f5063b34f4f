"""Chunkwise prefill on the GPU against the fp64 oracle, through the C ABI.

Small cases are compared element by element at sizes that span several 64-token
chunks and 16-token tiles with ragged tails; the full-size workloads are compared in
full (single long sequence) or on sampled (sequence, head) units.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_serving_02_gb300 import inputs, kda
from tests.gpu_util import assert_prefill_close, np64, oracle_units

pytestmark = pytest.mark.gpu


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_prefill(inp, cu=None, cu_host=True, o_dtype=torch.float32, S0="inp"):
    g = _cuda(inp)
    s0 = g["S0"] if S0 == "inp" else S0
    cu_d = None if cu is None else torch.tensor(cu, dtype=torch.int32, device="cuda")
    cu_h = None if (cu is None or not cu_host) else torch.tensor(cu, dtype=torch.int32)
    o, S = kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=s0,
                                 cu_seqlens=cu_d, cu_seqlens_host=cu_h, o_dtype=o_dtype)
    torch.cuda.synchronize()
    return o.cpu(), S.cpu()


def test_tiny_config():
    """B=1, T=256, H=2, zero initial state: four chunks, every output compared."""
    inp = inputs.prefill_inputs(256, 2, 1, seed=0)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"])
    for dt in (torch.float32, torch.bfloat16):
        o, S = gpu_prefill(inp, o_dtype=dt)
        assert o.dtype == dt
        assert_prefill_close(o, S, o_ref, S_ref, "tiny %s" % dt)


@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 130, 200])
def test_dense_batch_ragged_lengths(T):
    B, H = 2, 3
    inp = inputs.prefill_inputs(B * T, H, B, seed=10 + T, init_state=True, batch_rows=B)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    o, S = gpu_prefill(inp)
    assert_prefill_close(o, S, o_ref, S_ref, "T=%d" % T)


@pytest.mark.parametrize("cu_host", [True, False])
def test_packed_varlen_with_empty_and_short_sequences(cu_host):
    lens = [0, 1, 64, 100, 300, 17, 0, 129]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    H = 2
    inp = inputs.prefill_inputs(cu[-1], H, len(lens), seed=3, init_state=True)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu, cu_host=cu_host)
    assert_prefill_close(o, S, o_ref, S_ref, "varlen")
    for n, L in enumerate(lens):
        if L == 0:
            assert torch.equal(S[n], inp["S0"][n]), "an empty sequence must return its initial state"


def test_packed_equals_separate_runs():
    """Chunks restart at every sequence start, so a packed batch gives each sequence
    exactly the result of running it alone."""
    lens = [70, 5, 128]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    H = 3
    inp = inputs.prefill_inputs(cu[-1], H, len(lens), seed=4, init_state=True)
    o, S = gpu_prefill(inp, cu=cu)
    for n in range(len(lens)):
        a, e = cu[n], cu[n + 1]
        part = {k: (v[:, a:e].contiguous() if k in ("q", "k", "v", "z", "b") else v) for k, v in inp.items()}
        part["S0"] = inp["S0"][n:n + 1].contiguous()
        on, Sn = gpu_prefill(part)
        assert torch.equal(on[0], o[0, a:e]) and torch.equal(Sn[0], S[n]), "sequence %d" % n


def test_head_permutation_equivariance():
    T, H = 150, 4
    inp = inputs.prefill_inputs(T, H, 1, seed=6, init_state=True)
    o, S = gpu_prefill(inp)
    perm = [2, 0, 3, 1]
    pinp = {k: (v[..., perm, :].contiguous() if k in ("q", "k", "v", "z") else v) for k, v in inp.items()}
    pinp["b"] = inp["b"][..., perm].contiguous()
    pinp["A"] = inp["A"][perm].contiguous()
    pinp["S0"] = inp["S0"][:, perm].contiguous()
    op, Sp = gpu_prefill(pinp)
    assert torch.equal(op, o[..., perm, :]) and torch.equal(Sp, S[:, perm])


def test_no_decay_no_write_keeps_state():
    """z = -inf gives a = 1 exactly and b = -inf gives beta = 0: the state passes
    through unchanged and o_t = S0^T q_t."""
    T, H = 130, 2
    inp = inputs.prefill_inputs(T, H, 1, seed=7, init_state=True)
    inp["z"] = torch.full_like(inp["z"], -float("inf"))
    inp["b"] = torch.full_like(inp["b"], -float("inf"))
    o, S = gpu_prefill(inp)
    assert torch.equal(S, inp["S0"]), "state must pass through bit-identical"
    o_ref = np.einsum("thc,hcj->thj", np64(inp["q"][0]), np64(inp["S0"][0]))
    assert_prefill_close(o[0], None, o_ref, None, "identity")


def test_strongest_decay_everywhere():
    """z = +inf puts every token at the decay bound log a = -5: inside a 64-token chunk the
    decay spans e^-315, and the tile factors reach e^75; nothing may overflow."""
    T, H = 200, 2
    inp = inputs.prefill_inputs(T, H, 1, seed=8, init_state=True)
    inp["z"] = torch.full_like(inp["z"], float("inf"))
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    o, S = gpu_prefill(inp)
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    assert_prefill_close(o, S, o_ref, S_ref, "decay bound")


def _decay_pattern(inp, start, moderate=0.5):
    """z on every chunk position p = t mod 64: the bound decay (z = +inf, log a = -5
    exactly) on p in [start, start + 16), a moderate decay on the 16 positions before
    (log a between -0.4 and -0.6 across the channels, so that 16 tokens sum to about
    -6.4 .. -9.6), and no decay (z = -inf, a = 1) elsewhere."""
    z = inp["z"]
    T, H = z.shape[1], z.shape[2]
    p = torch.arange(T) % 64
    eA = torch.exp(inp["A"].double())                          # [H]
    f = 0.8 + 0.4 * torch.arange(128, dtype=torch.float64) / 127  # per channel
    frac = moderate / 5.0 * f                                   # sigmoid value giving log a = -moderate f
    zmod = (torch.log(frac / (1 - frac))[None, :] / eA[:, None]).float()  # [H, 128]
    out = torch.full_like(z, -float("inf"))
    bound = ((p >= start) & (p < start + 16))
    mod = ((p >= start - 16) & (p < start)) | ((p - 64 >= start - 16) & (p - 64 < start))
    out[0, bound] = float("inf")
    out[0, mod] = zmod
    inp["z"] = out
    return inp


@pytest.mark.parametrize("start", [1, 17, 33, 48])
def test_bound_decay_next_to_a_moderate_run(start):
    """Sixteen tokens at the decay bound right after sixteen of moderate decay, no decay
    elsewhere: the factors of the decayed Gram products around a reference token reach
    e^80 on one side while the other side's factor approaches the fp32/bf16 underflow
    (about e^-87), which is where a factoring that lets one factor exceed 1 while the
    other underflows would lose products of size e^-7 ('From Linear Attention to KDA',
    §5.4 bounded decay, §8 tiles). Element by element against the oracle, at several
    positions of the pattern within the 64-token chunk."""
    T, H = 200, 2
    inp = _decay_pattern(inputs.prefill_inputs(T, H, 1, seed=14 + start, init_state=True), start)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    o, S = gpu_prefill(inp)
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    assert_prefill_close(o, S, o_ref, S_ref, "decay pattern at %d" % start)


def test_full_write_strength_retrieves_the_last_value():
    """b = +inf gives beta = 1 exactly on every token. The delta rule then makes the last
    key retrieve its value: S_T^T k_T = v_T up to the deviation of ||k_T|| from 1 (k is
    normalised in fp32, then rounded to bf16). S_T^T k_T is compared with the oracle's,
    and o and S element by element ('From Linear Attention to KDA', §5.1)."""
    T, H = 150, 2
    inp = inputs.prefill_inputs(T, H, 1, seed=15, init_state=True)
    inp["b"] = torch.full_like(inp["b"], float("inf"))
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    o, S = gpu_prefill(inp)
    assert_prefill_close(o, S, o_ref, S_ref, "beta = 1")
    k_last = np64(inp["k"][0, T - 1])                       # [H, 128]
    v_last = np64(inp["v"][0, T - 1])
    r_gpu = np.einsum("hcj,hc->hj", np64(S[0]), k_last)
    r_ref = np.einsum("hcj,hc->hj", S_ref[0], k_last)
    rms = float(np.sqrt(np.mean(r_ref ** 2)))
    assert np.max(np.abs(r_gpu - r_ref)) <= 5e-3 * rms
    # the oracle itself retrieves v_T to the bf16 norm error of k_T
    assert np.max(np.abs(r_ref - v_last)) <= 2e-2 * float(np.sqrt(np.mean(v_last ** 2)))


def test_invalid_device_cu_seqlens_is_reported():
    """Without a host copy, a falling cu_seqlens is caught on the device: the workspace
    status says so, final_state is NaN and o is left untouched."""
    cu = [0, 100, 50, 256]
    H = 2
    inp = _cuda(inputs.prefill_inputs(256, H, 3, seed=9, init_state=True))
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o = torch.full(inp["q"].shape, 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(256, 3, H), dtype=torch.uint8, device="cuda")
    _, S = kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                                 initial_state=inp["S0"], cu_seqlens=cu_d, o=o, workspace=ws)
    assert kda.kda_workspace_status(ws) == -4
    assert torch.isnan(S).all()
    assert (o == 7.0).all()
    # the same workspace then serves a valid call and reports ok
    cu_d = torch.tensor([0, 50, 100, 256], dtype=torch.int32, device="cuda")
    kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                          initial_state=inp["S0"], cu_seqlens=cu_d, o=o, workspace=ws)
    assert kda.kda_workspace_status(ws) == 0


def test_host_cu_seqlens_rejected_before_launch():
    H = 2
    inp = _cuda(inputs.prefill_inputs(256, H, 3, seed=9))
    cu_d = torch.tensor([0, 100, 50, 256], dtype=torch.int32, device="cuda")
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_chunk_prefill(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], cu_seqlens=cu_d,
                              cu_seqlens_host=cu_d.cpu())
    assert ei.value.status == -4


def test_prefill_then_decode_equals_longer_prefill():
    """The chunked and the recurrent path agree on the state ('Kimi K3' page: both
    paths must give the same state-update semantics)."""
    T, m, H = 200, 9, 3
    inp = inputs.prefill_inputs(T + m, H, 1, seed=11, init_state=True)
    g = _cuda(inp)
    o_long, S_long = kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"],
                                           initial_state=g["S0"], o_dtype=torch.float32)
    head = {k: (v[:, :T].contiguous() if k in ("q", "k", "v", "z", "b") else v) for k, v in g.items()}
    o1, S = kda.kda_chunk_prefill(head["q"], head["k"], head["v"], head["z"], head["A"], head["b"],
                                  initial_state=g["S0"], o_dtype=torch.float32)
    state = S.clone()
    outs = [o1[0]]
    for t in range(T, T + m):
        ot = kda.kda_recurrent_decode(g["q"][:, t].contiguous(), g["k"][:, t].contiguous(), g["v"][:, t].contiguous(),
                                      g["z"][:, t].contiguous(), g["A"], g["b"][:, t].contiguous(), state)
        outs.append(ot)
    o_split = torch.cat(outs, 0)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    assert_prefill_close(o_split.cpu(), state.cpu(), o_ref[0], S_ref, "prefill + decode vs oracle")
    assert_prefill_close(o_split.cpu(), state.cpu(), np64(o_long[0]), np64(S_long), "prefill + decode vs long")


@pytest.mark.parametrize("lens,H", [([4000, 2000, 0, 900], 2), ([2000], 1), ([1700, 3000], 3),
                                    ([8000, 150, 0, 256, 257], 2)])
def test_segmented_walk(lens, H):
    """Few long sequences take the segmented walk: per-segment affine state maps from
    walks started at zero and at the identity, chained per sequence, then every segment
    walked again from its true input state. Ragged segment tails and an empty sequence
    included; in the last case the segments are 4 chunks long, so the 150- and 256-token
    sequences are one segment each (their whole walk runs in the first phase) and the
    257-token one ends in a one-chunk segment."""
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    inp = inputs.prefill_inputs(cu[-1], H, len(lens), seed=13, init_state=True)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu)
    assert_prefill_close(o, S, o_ref, S_ref, "segmented %s" % lens)


@pytest.mark.parametrize("seed", range(6))
def test_segmented_walk_random(seed):
    """Random batches that take the segmented walk (checked through the launch count):
    one to four sequences, lengths chunk-aligned or ragged, with an occasional empty or
    short one, against the oracle."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 5))
    H = int(rng.integers(1, 4))
    lens = []
    for _ in range(n):
        kind = rng.integers(0, 4)
        if kind == 0:
            lens.append(int(rng.integers(24, 80)) * 64)          # whole chunks
        elif kind == 1:
            lens.append(int(rng.integers(1600, 5000)))          # ragged tail
        elif kind == 2 and n > 1:
            lens.append(int(rng.integers(0, 3)) * int(rng.integers(1, 70)))  # empty or short
        else:
            lens.append(int(rng.integers(2000, 4000)))
    total = int(sum(lens))
    if kda.kda_chunk_prefill_walk_form(total, n, H) == 0:
        lens[0] += 64 * 24 * n  # long enough on average for the segmented walk
        total = int(sum(lens))
    assert kda.kda_chunk_prefill_walk_form(total, n, H) in (1, 2), (lens, H)
    assert kda.kda_chunk_prefill_launch_count(total, n, H) == 5
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    inp = inputs.prefill_inputs(total, H, n, seed=200 + seed, init_state=True)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu)
    assert_prefill_close(o, S, o_ref, S_ref, "segmented random %s x %d" % (lens, H))


def _slow_memory(inp, log_a=0.001, b_mean=-3.0, seed=0):
    """Weak decay and weak writes, so that the state keeps its memory over many chunks:
    z set per channel for log a = -log_a f (f from 0.5 to 1.5 over the channels), b around
    b_mean (beta about 0.05). The synthetic default decays by about e^-160 per chunk, which
    leaves every segment map M of the segmented walk at zero; here M is far from it."""
    T, H = inp["z"].shape[1], inp["z"].shape[2]
    eA = torch.exp(inp["A"].double())
    f = 0.5 + torch.arange(128, dtype=torch.float64) / 127
    frac = log_a / 5.0 * f
    z = (torch.log(frac / (1 - frac))[None, :] / eA[:, None]).float()
    inp["z"] = z[None, None].expand(1, T, H, 128).contiguous()
    g = torch.Generator().manual_seed(seed)
    inp["b"] = (b_mean + 0.5 * torch.randn(inp["b"].shape, generator=g)).float()
    return inp


@pytest.mark.parametrize("lens,H,form", [([3000, 1800], 2, 1), ([5000], 1, 1), ([10240, 10000, 10480], 5, 2)])
def test_segmented_walk_slow_memory(lens, H, form):
    """The segmented walk where the segment maps matter: with weak decay and weak writes
    the map M of a segment (its state from the identity) stays of order one, so the
    products M S_in carry the state from segment to segment ('From Linear Attention to
    KDA', §7.5). Both forms: each output walk chaining the maps before it on the tensor
    cores (form 1; [5000] x 1 cuts ten segments, so the last one chains eight maps),
    and the combine kernel (form 2: 3 sequences x 5 heads in 32-segment tables).
    Against the oracle, element by element."""
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    n = len(lens)
    assert kda.kda_chunk_prefill_walk_form(cu[-1], n, H) == form, (lens, H)
    inp = _slow_memory(inputs.prefill_inputs(cu[-1], H, n, seed=31, init_state=True), seed=32)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu)
    assert_prefill_close(o, S, o_ref, S_ref, "segmented, slow memory %s" % lens)


@pytest.mark.parametrize("lens,H,E,init", [([10240, 10000, 10480], 5, 2, True), ([14000, 2000, 14720], 5, 3, False)])
def test_segmented_walk_long_ends(lens, H, E, init):
    """The combine form with long end segments, forced through the test hook on batches
    small enough for the oracle (the sizes choose them only for much longer chains): the
    first and last segment of each long enough sequence E segment lengths long, the
    walks of both phases listed longest first with heads as the fastest grid index. In the
    second batch the 2000-token sequence is too short for long ends and keeps the uniform
    cut. Weak decay and writes, so the maps carry the state; against the oracle, and the
    cut must change the rounding against the uniform one."""
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    n = len(lens)
    assert kda.kda_chunk_prefill_walk_form(cu[-1], n, H) == 2, (lens, H)
    inp = _slow_memory(inputs.prefill_inputs(cu[-1], H, n, seed=37, init_state=init), seed=38)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"],
                                      S0=inp["S0"] if init else None, cu_seqlens=cu)
    o1, S1 = gpu_prefill(inp, cu=cu, S0="inp" if init else None)
    kda.kda_debug_segment_ends(E)
    try:
        o, S = gpu_prefill(inp, cu=cu, S0="inp" if init else None)
    finally:
        kda.kda_debug_segment_ends(0)
    assert_prefill_close(o, S, o_ref, S_ref, "segmented, long ends E=%d %s" % (E, lens))
    assert not torch.equal(S, S1)


@pytest.mark.parametrize("T,B,H", [(4096, 2, 12), (8192, 2, 6)])
def test_dense_segmented_walk_defers_intra_items(T, B, H):
    """Dense batches in the chained form whose intra-chunk items pass a whole number of
    rounds of the GPU's SMs: the items past k * SMs - 1 (the last chunks of the last
    sequence, read only by its last output walk) run in a second intra-chunk launch beside
    the map walk. o, final_state and the workspace start as NaN bytes, so an output walk
    that read a record before that launch wrote it would show; against the oracle."""
    assert kda.kda_chunk_prefill_walk_form(B * T, B, H) == 1
    inp = inputs.prefill_inputs(B * T, H, B, seed=41, init_state=True, batch_rows=B)
    g = _cuda(inp)
    o = torch.full(tuple(inp["q"].shape), float("nan"), dtype=torch.float32, device="cuda")
    S = torch.full((B, H, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.full((kda.kda_chunk_prefill_workspace_size(B * T, B, H),), 0xFF, dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=g["S0"], o=o,
                          final_state=S, workspace=ws, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"])
    assert_prefill_close(o.cpu(), S.cpu(), o_ref, S_ref, "dense %d x %d x %d" % (B, T, H))


@pytest.mark.parametrize("lens,H,form", [([3000, 1800], 2, 1), ([10240, 10000, 10480], 5, 2)])
def test_segmented_walk_without_initial_state(lens, H, form):
    """Both segmented forms with no initial state (zero): segment 0 starts from zero in
    both phases, every later segment from what the maps carry. Weak decay and writes, so
    the maps matter; against the oracle."""
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    n = len(lens)
    assert kda.kda_chunk_prefill_walk_form(cu[-1], n, H) == form, (lens, H)
    inp = _slow_memory(inputs.prefill_inputs(cu[-1], H, n, seed=35), seed=36)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu, S0=None)
    assert_prefill_close(o, S, o_ref, S_ref, "segmented, no initial state %s" % lens)


def test_plain_walk_slow_memory():
    """The same weak decay and writes on the plain walk (many chains), 1,500 tokens."""
    lens = [1500] * 40
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    assert kda.kda_chunk_prefill_launch_count(cu[-1], len(lens), 2) == 3
    inp = _slow_memory(inputs.prefill_inputs(cu[-1], 2, len(lens), seed=33, init_state=True), seed=34)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu)
    assert_prefill_close(o, S, o_ref, S_ref, "plain, slow memory")


@pytest.mark.parametrize("seed", range(4))
def test_plain_walk_random(seed):
    """Random batches of many short sequences (one plain walk unit per chain, checked
    through the launch count), lengths drawn from the edge values 0, 1, 63, 64, 65 and
    from 1 .. 700, against the oracle."""
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(8, 41))
    H = int(rng.integers(1, 5))
    edges = [0, 1, 63, 64, 65]
    lens = [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 701)) for _ in range(n)]
    total = int(sum(lens))
    assert kda.kda_chunk_prefill_launch_count(total, n, H) == 3, (lens, H)
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    inp = inputs.prefill_inputs(total, H, n, seed=400 + seed, init_state=True)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu)
    assert_prefill_close(o, S, o_ref, S_ref, "plain random %d sequences x %d" % (n, H))


@pytest.mark.parametrize("n", [1024, 1100])
def test_plain_walk_many_sequences(n):
    """The plain walk's unit order: up to 1024 sequences are listed longest first (the plan
    kernel's sort, padded to a power of two), more are left in sequence order; lengths
    0 .. 200 with ties, one head, against the oracle."""
    rng = np.random.default_rng(500 + n)
    lens = [int(x) for x in rng.choice([0, 1, 5, 64, 65, 130, 200], size=n)]
    total = int(sum(lens))
    assert kda.kda_chunk_prefill_launch_count(total, n, 1) == 3
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    inp = inputs.prefill_inputs(total, 1, n, seed=600 + n, init_state=True)
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    o, S = gpu_prefill(inp, cu=cu)
    assert_prefill_close(o, S, o_ref, S_ref, "plain walk, %d sequences" % n)


@pytest.mark.parametrize("lens,H,o_dtype", [([300, 0, 1, 64, 129], 3, torch.bfloat16),   # plain walk
                                            ([5000, 0, 1700], 2, torch.float32),       # segmented, chained
                                            ([10240, 10000, 10480], 5, torch.bfloat16)])  # segmented, combine
def test_every_output_written_over_poison(lens, H, o_dtype):
    """o, final_state and the workspace start filled with NaN bytes: every output must be
    written (finite) and right, and nothing may read workspace that was not written."""
    total = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    inp = inputs.prefill_inputs(total, H, len(lens), seed=500, init_state=True)
    g = _cuda(inp)
    o = torch.full((1, total, H, 128), float("nan"), dtype=o_dtype, device="cuda")
    S = torch.full((len(lens), H, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.full((kda.kda_chunk_prefill_workspace_size(total, len(lens), H),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    kda.kda_chunk_prefill(g["q"], g["k"], g["v"], g["z"], g["A"], g["b"], initial_state=g["S0"],
                          cu_seqlens=torch.tensor(cu, dtype=torch.int32, device="cuda"),
                          cu_seqlens_host=torch.tensor(cu, dtype=torch.int32), o=o, final_state=S, workspace=ws,
                          o_dtype=o_dtype)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
    o_ref, S_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["b"], S0=inp["S0"],
                                      cu_seqlens=cu)
    assert_prefill_close(o.cpu(), S.cpu(), o_ref, S_ref, "poisoned %s" % lens)
