"""Seeded synthetic inputs for KDA prefill and decode.

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the method's arithmetic. The tests and the benchmark
hand the same tensors to the CUDA path and to the CPU oracle.

Recipe (every tensor from one torch.Generator seeded with `seed`, drawn in the
order q, k, v, z, A, b, S0):
  q, k  ~ N(0, 1) [.., H, d_k], L2-normalised over d_k in fp32, then cast to bf16
        (the model normalises q and k before the operator: 'From Linear Attention to
        KDA', §5.3; so ||k|| = 1 only to bf16 rounding)
  v     ~ N(0, 1) [.., H, d_v] cast to bf16
  z     ~ N(0, 1) [.., H, d_k] fp32 (raw decay pre-activation)
  A_h   = log U(1, 16) [H] fp32
  b     ~ N(0, 1) [.., H] fp32 (raw write-strength pre-activation)
  S0    = 0, or ~ N(0, 0.02^2) [N, H, d_k, d_v] fp32
Packed varlen lengths are integers drawn uniformly in [lo, hi] from their own
generator seeded with `seed`.
"""
import torch

D = 128


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _unit_bf16(x):
    return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)


def varlen_lengths(n_seqs, lo, hi, seed=0):
    """n_seqs sequence lengths, uniform integers in [lo, hi]."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n_seqs,), generator=g).tolist()


def cu_seqlens_from_lengths(lengths, device="cpu"):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def prefill_inputs(T_total, H, n_seqs, seed=0, init_state=False, state_std=0.02,
                   d_k=D, d_v=D, device="cpu", batch_rows=1):
    """Inputs of one prefill call.

    Tokens are laid out [batch_rows, T_total // batch_rows, H, d] (batch_rows = B of a
    dense batch, 1 for a packed varlen batch). Returns a dict with q, k, v (bf16),
    z, A, b (fp32) and S0 (fp32 [n_seqs, H, d_k, d_v] or None).
    """
    assert T_total % batch_rows == 0
    g = _gen(seed, device)
    shp = (batch_rows, T_total // batch_rows, H)
    f32 = torch.float32
    q = _unit_bf16(torch.randn(shp + (d_k,), generator=g, device=device, dtype=f32))
    k = _unit_bf16(torch.randn(shp + (d_k,), generator=g, device=device, dtype=f32))
    v = torch.randn(shp + (d_v,), generator=g, device=device, dtype=f32).to(torch.bfloat16)
    z = torch.randn(shp + (d_k,), generator=g, device=device, dtype=f32)
    A = torch.log(1.0 + 15.0 * torch.rand((H,), generator=g, device=device, dtype=f32))
    b = torch.randn(shp, generator=g, device=device, dtype=f32)
    S0 = None
    if init_state:
        S0 = state_std * torch.randn((n_seqs, H, d_k, d_v), generator=g, device=device, dtype=f32)
    return dict(q=q, k=k, v=v, z=z, A=A, b=b, S0=S0)


def decode_state(N, H, seed=0, state_std=0.02, d_k=D, d_v=D, device="cpu"):
    """Initial per-sequence recurrent states ~ N(0, state_std^2), fp32 [N, H, d_k, d_v]."""
    g = _gen(seed, device)
    return state_std * torch.randn((N, H, d_k, d_v), generator=g, device=device, dtype=torch.float32)


def decode_step_inputs(N, H, seed=0, step=0, d_k=D, d_v=D, device="cpu", A=None):
    """One decode step: q, k, v [N, H, d] bf16; z [N, H, d_k] fp32; b [N, H] fp32; A [H].

    Each step draws from its own generator (seed, step) so steps can be regenerated
    one at a time; A is drawn once per (seed) unless passed in.
    """
    g = _gen(seed * 1000003 + 7919 * (step + 1), device)
    f32 = torch.float32
    q = _unit_bf16(torch.randn((N, H, d_k), generator=g, device=device, dtype=f32))
    k = _unit_bf16(torch.randn((N, H, d_k), generator=g, device=device, dtype=f32))
    v = torch.randn((N, H, d_v), generator=g, device=device, dtype=f32).to(torch.bfloat16)
    z = torch.randn((N, H, d_k), generator=g, device=device, dtype=f32)
    b = torch.randn((N, H), generator=g, device=device, dtype=f32)
    if A is None:
        ga = _gen(seed * 1000003 + 1, device)
        A = torch.log(1.0 + 15.0 * torch.rand((H,), generator=ga, device=device, dtype=f32))
    return dict(q=q, k=k, v=v, z=z, A=A, b=b)


def fused_decode_params(H, seed=0, d=D, device="cpu"):
    """Synthetic stand-ins for the layer weights around the fused decode: conv taps
    fp32 [3, H, d, 4] ~ N(0, 0.5^2) and the RMSNorm weight fp32 [d] ~ 1 + N(0, 0.1^2)."""
    g = _gen(seed * 1000003 + 2, device)
    f32 = torch.float32
    conv_w = 0.5 * torch.randn((3, H, d, 4), generator=g, device=device, dtype=f32)
    norm_w = 1.0 + 0.1 * torch.randn((d,), generator=g, device=device, dtype=f32)
    return dict(conv_w=conv_w, norm_w=norm_w)


def fused_decode_step_inputs(N, H, seed=0, step=0, d=D, device="cpu"):
    """One fused decode token: the pre-conv projections x_q, x_k, x_v ~ N(0, 1) bf16
    [N, H, d], z ~ N(0, 1) fp32, b ~ N(0, 1) fp32 [N, H], the output-gate pre-activation
    g ~ N(0, 1) fp32 [N, H, d], and A [H] drawn once per seed as for decode."""
    gen = _gen(seed * 1000003 + 7919 * (step + 1) + 3, device)
    f32 = torch.float32
    xq, xk, xv = (torch.randn((N, H, d), generator=gen, device=device, dtype=f32).to(torch.bfloat16)
                  for _ in range(3))
    z = torch.randn((N, H, d), generator=gen, device=device, dtype=f32)
    b = torch.randn((N, H), generator=gen, device=device, dtype=f32)
    g = torch.randn((N, H, d), generator=gen, device=device, dtype=f32)
    ga = _gen(seed * 1000003 + 1, device)
    A = torch.log(1.0 + 15.0 * torch.rand((H,), generator=ga, device=device, dtype=f32))
    return dict(x_q=xq, x_k=xk, x_v=xv, z=z, A=A, b=b, g=g)
