"""Seeded synthetic inputs for the KDA core workloads.

Shared by the tests, the benchmark and the smoke check, and by both the CUDA
path and the oracle.  This module holds input distributions only -- none of
the KDA arithmetic.  Everything is drawn on the CPU from ``torch.Generator``
so that every machine sees the same bits; bf16 tensors are rounded once here.

Library layouts (row-major):
  q, k, g : [T_total, H, K]    v : [T_total, H, V]    beta : [T_total, H]
  states  : [N, H, V, K] fp32  (key dim contiguous)
  decode  : q, k, g [N, H, K]; v [N, H, V]; beta [N, H]; pool [slots, H, V, K]

Named workloads (seed in brackets):
  recurrence_small  B=1 H=2 T=256 K=V=128 fp32, g ~ U[-0.2,-0.001], S0 = 0   [0]
  prefill_4k        B=1 H=32 T=4096 bf16 q/k/v, g ~ U[-0.1,-0.0005], S0 = 0  [1]
  varlen_8          8 packed sequences, lengths ~ U{512..8192}, H=32 bf16,
                    g ~ U[-0.1,-0.0005], S0 ~ N(0, 0.02^2)                    [2]
  decode_256        256 seqs x H=32, pool N(0, 0.02^2), 64 steps of bf16 tokens [3]
  long_131k         B=1 H=32 T=131072 bf16, g per (t,h,k): 90% U[-0.01,-1e-5],
                    10% U[-3,-1]; then 256 decode steps                      [4]
q, k, v ~ N(0, 1); beta = sigmoid(N(0, 1)) (already activated), fp32.

Gated variants (the model's raw gates; the library activates them in-kernel):
  raw_gate [T, H, K] and raw_beta [T, H] ~ N(0, 1) in the q/k/v dtype,
  a_log [H] = log U[a_lo, a_hi] (the model initialises A_log = log U[1, 16]),
  dt_bias [H, K] ~ U[b_lo, b_hi] fp32, and an optional lower bound
  (the lower-bounded "safe" gate keeps every decay in (lower_bound, 0)).
  prefill_4k_gated  prefill_4k's q/k/v with raw gates, A_log = log U[1, 16],
                    dt_bias ~ U[-1, 1], lower bound -5                       [5]
Speculative decode: S draft tokens per sequence, q, k, g [N, S, H, K],
v [N, S, H, V], beta [N, S, H], drawn like decode tokens.
Short convolution: x [T, D = 3 H K] ~ N(0, 1), weight [ks = 4, D] ~ U[-1/2, 1/2]
(bf16 unless given); decode conv states [slots, ks - 1, D] ~ N(0, 1).
Output epilogue inputs: out_gate [T, H, V] ~ N(0, 1) in the q dtype, o_norm
weight [V] ~ U[0.5, 1.5] fp32, eps 1e-5.
"""
from __future__ import annotations

import torch

K_DIM = 128
V_DIM = 128


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(int(seed))


def _normal(shape, gen, std=1.0, dtype=torch.float32):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32) * std
    return x.to(dtype)


def _uniform(shape, gen, lo, hi):
    return torch.rand(*shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo


def _beta(shape, gen):
    return torch.sigmoid(torch.randn(*shape, generator=gen, dtype=torch.float32))


def decay_uniform(shape, gen, lo, hi):
    """Per-channel log-decay g ~ U[lo, hi] (all non-positive)."""
    return _uniform(shape, gen, lo, hi)


def decay_mixed(shape, gen, p_strong=0.1, weak=(-0.01, -1e-5), strong=(-3.0, -1.0)):
    """Each element independently: strong decay with probability p_strong, else weak."""
    w = _uniform(shape, gen, *weak)
    s = _uniform(shape, gen, *strong)
    pick = torch.rand(*shape, generator=gen) < p_strong
    return torch.where(pick, s, w)


def prefill(lengths, H=32, K=K_DIM, V=V_DIM, dtype=torch.bfloat16, seed=1,
            g_range=(-0.1, -0.0005), g_mixed=False, init_std=None, packed=True):
    """Packed prefill inputs for sequences of the given lengths.

    Returns a dict with q, k, v (dtype), g, beta (fp32), cu_seqlens (int32,
    [N+1]), initial_state ([N, H, V, K] fp32 or None), lengths.
    """
    lengths = [int(t) for t in lengths]
    T = sum(lengths)
    gen = _gen(seed)
    q = _normal((T, H, K), gen, dtype=dtype)
    k = _normal((T, H, K), gen, dtype=dtype)
    v = _normal((T, H, V), gen, dtype=dtype)
    if g_mixed:
        g = decay_mixed((T, H, K), gen)
    else:
        g = decay_uniform((T, H, K), gen, *g_range)
    beta = _beta((T, H), gen)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    s0 = None
    if init_std is not None:
        s0 = _normal((len(lengths), H, V, K), gen, std=init_std)
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu, initial_state=s0,
                lengths=lengths, H=H, K=K, V=V)


def varlen_lengths(n=8, lo=512, hi=8192, seed=2):
    gen = _gen(seed + 1000)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def decode_pool(n_slots, H=32, K=K_DIM, V=V_DIM, std=0.02, seed=3):
    """Pool of fp32 states [slots, H, V, K] ~ N(0, std^2)."""
    return _normal((n_slots, H, V, K), _gen(seed), std=std)


def decode_tokens(N, H=32, K=K_DIM, V=V_DIM, dtype=torch.bfloat16, seed=3, step=0,
                  g_range=(-0.1, -0.0005), g_mixed=False):
    """One decode token per sequence; a fresh seeded draw for every step."""
    gen = _gen(seed * 100003 + 7919 * (step + 1))
    q = _normal((N, H, K), gen, dtype=dtype)
    k = _normal((N, H, K), gen, dtype=dtype)
    v = _normal((N, H, V), gen, dtype=dtype)
    g = decay_mixed((N, H, K), gen) if g_mixed else decay_uniform((N, H, K), gen, *g_range)
    beta = _beta((N, H), gen)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def gate_params(H, K=K_DIM, seed=5, a_range=(1.0, 16.0), bias_range=(-1.0, 1.0)):
    """a_log [H] = log U[a_range], dt_bias [H, K] ~ U[bias_range], fp32."""
    gen = _gen(seed * 7 + 3)
    a_log = torch.log(_uniform((H,), gen, *a_range))
    dt_bias = _uniform((H, K), gen, *bias_range)
    return a_log, dt_bias


def with_raw_gates(x, seed=5, dtype=None, a_range=(1.0, 16.0), bias_range=(-1.0, 1.0),
                   lower_bound=-5.0):
    """Add raw gates and gate parameters to a prefill or decode input dict
    (raw_gate like g, raw_beta like beta, in the q dtype unless given)."""
    dtype = x["q"].dtype if dtype is None else dtype
    gen = _gen(seed * 13 + 11)
    y = dict(x)
    y["raw_gate"] = _normal(tuple(x["g"].shape), gen, dtype=dtype)
    y["raw_beta"] = _normal(tuple(x["beta"].shape), gen, dtype=dtype)
    H, K = x["g"].shape[-2], x["g"].shape[-1]
    y["a_log"], y["dt_bias"] = gate_params(H, K, seed, a_range, bias_range)
    y["lower_bound"] = lower_bound
    return y


def with_output_gate(x, seed=6, dtype=None, eps=1e-5):
    """Add the output epilogue's inputs: out_gate like v, o_norm weight [V], eps."""
    dtype = x["q"].dtype if dtype is None else dtype
    gen = _gen(seed * 17 + 5)
    y = dict(x)
    y["out_gate"] = _normal(tuple(x["v"].shape), gen, dtype=dtype)
    y["norm_weight"] = _uniform((x["v"].shape[-1],), gen, 0.5, 1.5)
    y["norm_eps"] = eps
    return y


def spec_tokens(N, S, H=32, K=K_DIM, V=V_DIM, dtype=torch.bfloat16, seed=7, step=0,
                g_range=(-0.1, -0.0005)):
    """S draft tokens per sequence for speculative decode: q, k, g [N, S, H, K],
    v [N, S, H, V], beta [N, S, H] (activated)."""
    gen = _gen(seed * 100019 + 104729 * (step + 1))
    q = _normal((N, S, H, K), gen, dtype=dtype)
    k = _normal((N, S, H, K), gen, dtype=dtype)
    v = _normal((N, S, H, V), gen, dtype=dtype)
    g = decay_uniform((N, S, H, K), gen, *g_range)
    beta = _beta((N, S, H), gen)
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def conv_inputs(lengths, D=3 * 32 * K_DIM, ks=4, dtype=torch.bfloat16, seed=8):
    """Short-conv inputs: x [T, D] ~ N(0, 1) (the fused q/k/v projection, D =
    3 H K), weight [ks, D] ~ U[-1/2, 1/2] (the model's kaiming-uniform bound for
    a fan-in of ks = 4), cu_seqlens [N+1] int32."""
    lengths = [int(t) for t in lengths]
    gen = _gen(seed * 31 + 17)
    x = _normal((sum(lengths), D), gen, dtype=dtype)
    w = _uniform((ks, D), gen, -0.5, 0.5).to(dtype)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return dict(x=x, weight=w, cu_seqlens=cu, lengths=lengths, ks=ks, D=D)


# ---- the named workloads ---------------------------------------------------

def recurrence_small():
    return prefill([256], H=2, dtype=torch.float32, seed=0, g_range=(-0.2, -0.001))


def prefill_4k(T=4096, H=32):
    return prefill([T], H=H, dtype=torch.bfloat16, seed=1)


def varlen_8(H=32, lengths=None):
    if lengths is None:
        lengths = varlen_lengths()
    return prefill(lengths, H=H, dtype=torch.bfloat16, seed=2, init_std=0.02)


def long_131k(T=131072, H=32):
    return prefill([T], H=H, dtype=torch.bfloat16, seed=4, g_mixed=True)


def prefill_4k_gated(T=4096, H=32):
    return with_raw_gates(prefill_4k(T, H), seed=5)


WORKLOADS = {
    "recurrence_small": "B=1 H=2 T=256 K=V=128 fp32, g~U[-0.2,-0.001], seed 0",
    "prefill_4k": "B=1 H=32 T=4096 K=V=128 bf16 q/k/v, g~U[-0.1,-0.0005], S0=0, seed 1",
    "varlen_8": "8 packed seqs, lengths U{512..8192}, H=32 bf16, S0~N(0,0.02^2), seed 2",
    "decode_256": "256 seqs x H=32, pool fp32 [256,32,128,128]~N(0,0.02^2), 64 bf16 steps, seed 3",
    "long_131k": "B=1 H=32 T=131072 bf16, g 90% U[-0.01,-1e-5] / 10% U[-3,-1], +256 decode steps, seed 4",
    "prefill_4k_gated": "prefill_4k with raw bf16 gates ~N(0,1), A_log=log U[1,16], dt_bias~U[-1,1], lower bound -5, seed 5",
}
