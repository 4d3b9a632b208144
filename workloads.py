"""Seeded synthetic inputs for the five broadcast workloads.

This module only draws and lays out inputs: it holds none of the operators'
arithmetic, and both the CUDA path's tests and the CPU oracle read the same
host tensors it returns.  Every tensor comes from
``torch.Generator('cpu').manual_seed(seed)`` in the order listed for each
workload; N(mu, sigma) is ``randn * sigma + mu`` and U(lo, hi) is
``rand * (hi - lo) + lo``.

Workloads (default sizes; every size can be overridden for small parity
cases with the same structure):

* ``c1`` mul, a [P,M,Q] N(0,1) * b [M,1] N(0,1), g N(0,1)            (32,64,128)
* ``c2`` bias add, x [R,C] N(0,1) + bias [C] N(0,0.02), g N(0,1)        (4096,1024)
* ``c3`` affine, y1 = x[B,T,C] * gamma[C] U(0.5,1.5); y2 = y1 + beta[C]
  N(0,0.1); g N(0,1)                                                    (16,1024,768)
* ``c4`` attention scores, t = scores[N,H,T,T] N(0,1) + mask[1,1,T,T]
  (0 where j <= i, -1e9 above the diagonal); out = t / scalar[1] (= 8.0);
  g N(0,1)                                                              (8,12,1024,1024)
* ``c5a`` a = storage[P,Q,M].transpose(1,2) -> [P,M,Q] (strides
  [Q*M, 1, M]), storage N(0,1); b [1,M,1] N(0,1); out = a - b; g N(0,1)   (128,256,512)
* ``c5b`` 8-d div: a [4,1,8,1,16,1,32,64] N(0,1); b = s*u with
  u U(0.5,1.5) [1,6,1,12,1,10,1,64] and s = 2*randint(0,2)-1 drawn after u;
  g N(0,1) of the broadcast shape [4,6,8,12,16,10,32,64]
* ``x1`` same-shape contiguous add, a [R,C] N(0,1) + b [R,C] N(0,1), g N(0,1)
  (4096,4096): a supplementary case for the contiguous path without
  broadcasting (not one of the five workloads of the benchmark step)
* ``u1`` unary ops on an FFN hidden activation, x [R,C] N(0,1), g N(0,1)
  (16384, 3072): GeLU forward and backward, then scale by 0.125 forward and
  backward (supplementary, outside the benchmark step)
* ``c4h``: ``c4`` with every tensor stored as bfloat16 (the same draws,
  rounded to bf16 by the caller; see ``BF16``), supplementary
* ``u1h``: ``u1`` stored as bfloat16 in the same way, supplementary
* ``c3f`` and ``c4f``: the inputs of ``c3`` and ``c4`` (same seeds and
  sizes), run as one fused two-op chain each, (x * gamma) + beta and
  (scores + mask) / scalar (supplementary, outside the benchmark step)

Each workload also lists its op steps (forward chain, then backward in
reverse) as data: ``("fwd", op, a_name, b_name, out_name)`` and
``("bwd", op, g_name, a_name, b_name, grad_a_name, grad_b_name)``; a fused
chain is ``("cfwd", op1, op2, a_name, b_name, c_name, out_name)`` and
``("cbwd", op1, op2, g_name, a_name, b_name, c_name, grad_a_name,
grad_b_name, grad_c_name)``; a unary op ``("ufwd", op, alpha, x_name,
out_name)`` and ``("ubwd", op, alpha, g_name, x_name, grad_x_name)``.
"""
from __future__ import annotations

import torch

SEEDS = {"c1": 1001, "c2": 1002, "c3": 1003, "c4": 1004, "c5a": 1005, "c5b": 1006, "x1": 1007,
         "u1": 1008}
# Fused-chain and bf16 workloads draw the inputs of the workload they derive from.
BASE = {"c3f": "c3", "c4f": "c4", "c4h": "c4", "u1h": "u1"}
# Workloads whose tensors are stored as bfloat16.
BF16 = {"c4h", "u1h"}

DEFAULT_DIMS = {
    "c1": dict(P=32, M=64, Q=128),
    "c2": dict(R=4096, C=1024),
    "c3": dict(B=16, T=1024, C=768),
    "c4": dict(N=8, H=12, T=1024),
    "c5a": dict(P=128, M=256, Q=512),
    "c5b": dict(a=(4, 1, 8, 1, 16, 1, 32, 64), b=(1, 6, 1, 12, 1, 10, 1, 64)),
    "x1": dict(R=4096, C=4096),
    "u1": dict(R=16384, C=3072),
}

# Forward chain then backward steps, in execution order.
STEPS = {
    "c1": [("fwd", "mul", "a", "b", "out"),
           ("bwd", "mul", "g", "a", "b", "grad_a", "grad_b")],
    "c2": [("fwd", "add", "x", "bias", "out"),
           ("bwd", "add", "g", "x", "bias", "grad_x", "grad_bias")],
    "c3": [("fwd", "mul", "x", "gamma", "y1"),
           ("fwd", "add", "y1", "beta", "y2"),
           ("bwd", "add", "g", "y1", "beta", "grad_y1", "grad_beta"),
           ("bwd", "mul", "grad_y1", "x", "gamma", "grad_x", "grad_gamma")],
    "c4": [("fwd", "add", "scores", "mask", "t"),
           ("fwd", "div", "t", "scalar", "out"),
           ("bwd", "div", "g", "t", "scalar", "grad_t", "grad_scalar"),
           ("bwd", "add", "grad_t", "scores", "mask", "grad_scores", "grad_mask")],
    "c5a": [("fwd", "sub", "a", "b", "out"),
            ("bwd", "sub", "g", "a", "b", "grad_a", "grad_b")],
    "c5b": [("fwd", "div", "a", "b", "out"),
            ("bwd", "div", "g", "a", "b", "grad_a", "grad_b")],
    "x1": [("fwd", "add", "a", "b", "out"),
           ("bwd", "add", "g", "a", "b", "grad_a", "grad_b")],
    "u1": [("ufwd", "gelu", 1.0, "x", "h"),
           ("ufwd", "scale", 0.125, "x", "s"),
           ("ubwd", "scale", 0.125, "g", "x", "grad_s"),
           ("ubwd", "gelu", 1.0, "g", "x", "grad_x")],
    "u1h": [("ufwd", "gelu", 1.0, "x", "h"),
            ("ufwd", "scale", 0.125, "x", "s"),
            ("ubwd", "scale", 0.125, "g", "x", "grad_s"),
            ("ubwd", "gelu", 1.0, "g", "x", "grad_x")],
    "c4h": [("fwd", "add", "scores", "mask", "t"),
            ("fwd", "div", "t", "scalar", "out"),
            ("bwd", "div", "g", "t", "scalar", "grad_t", "grad_scalar"),
            ("bwd", "add", "grad_t", "scores", "mask", "grad_scores", "grad_mask")],
    "c3f": [("cfwd", "mul", "add", "x", "gamma", "beta", "y2"),
            ("cbwd", "mul", "add", "g", "x", "gamma", "beta", "grad_x", "grad_gamma", "grad_beta")],
    "c4f": [("cfwd", "add", "div", "scores", "mask", "scalar", "out"),
            ("cbwd", "add", "div", "g", "scores", "mask", "scalar", "grad_scores", "grad_mask",
             "grad_scalar")],
}

NAMES = list(STEPS)

CAUSAL_MASK_VALUE = -1e9  # exactly representable in binary32


def _normal(gen, shape, mu=0.0, sigma=1.0):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * sigma + mu


def _uniform(gen, shape, lo, hi):
    return torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo


def _broadcast_dims(sa, sb):
    # Output shape of two same-rank shapes where each pair is equal or has a 1;
    # only used to size g for c5b (the shapes are fixed by the workload).
    return tuple(max(x, y) for x, y in zip(sa, sb))


def make_inputs(name: str, seed: int | None = None, **dims) -> dict:
    """Host (CPU) float32 input tensors of workload ``name``.

    ``dims`` overrides the default sizes (see ``DEFAULT_DIMS``) for small
    parity cases; ``seed`` overrides the workload's seed.
    """
    name = BASE.get(name, name)
    d = dict(DEFAULT_DIMS[name])
    d.update(dims)
    gen = torch.Generator("cpu").manual_seed(SEEDS[name] if seed is None else seed)
    if name == "c1":
        P, M, Q = d["P"], d["M"], d["Q"]
        a = _normal(gen, (P, M, Q))
        b = _normal(gen, (M, 1))
        g = _normal(gen, (P, M, Q))
        return dict(a=a, b=b, g=g)
    if name == "c2":
        R, C = d["R"], d["C"]
        x = _normal(gen, (R, C))
        bias = _normal(gen, (C,), 0.0, 0.02)
        g = _normal(gen, (R, C))
        return dict(x=x, bias=bias, g=g)
    if name == "c3":
        B, T, C = d["B"], d["T"], d["C"]
        x = _normal(gen, (B, T, C))
        gamma = _uniform(gen, (C,), 0.5, 1.5)
        beta = _normal(gen, (C,), 0.0, 0.1)
        g = _normal(gen, (B, T, C))
        return dict(x=x, gamma=gamma, beta=beta, g=g)
    if name == "c4":
        N, H, T = d["N"], d["H"], d["T"]
        scores = _normal(gen, (N, H, T, T))
        i = torch.arange(T).view(T, 1)
        j = torch.arange(T).view(1, T)
        mask = torch.where(j <= i, torch.tensor(0.0), torch.tensor(CAUSAL_MASK_VALUE))
        mask = mask.to(torch.float32).view(1, 1, T, T).contiguous()
        scalar = torch.tensor([8.0], dtype=torch.float32)
        g = _normal(gen, (N, H, T, T))
        return dict(scores=scores, mask=mask, scalar=scalar, g=g)
    if name == "c5a":
        P, M, Q = d["P"], d["M"], d["Q"]
        storage = _normal(gen, (P, Q, M))
        a = storage.transpose(1, 2)  # [P, M, Q], strides [Q*M, 1, M]
        b = _normal(gen, (1, M, 1))
        g = _normal(gen, (P, M, Q))
        return dict(a=a, b=b, g=g)
    if name == "c5b":
        sa, sb = tuple(d["a"]), tuple(d["b"])
        a = _normal(gen, sa)
        u = _uniform(gen, sb, 0.5, 1.5)
        s = (2 * torch.randint(0, 2, sb, generator=gen) - 1).to(torch.float32)
        b = s * u
        g = _normal(gen, _broadcast_dims(sa, sb))
        return dict(a=a, b=b, g=g)
    if name == "u1":
        R, C = d["R"], d["C"]
        x = _normal(gen, (R, C))
        g = _normal(gen, (R, C))
        return dict(x=x, g=g)
    if name == "x1":
        R, C = d["R"], d["C"]
        a = _normal(gen, (R, C))
        b = _normal(gen, (R, C))
        g = _normal(gen, (R, C))
        return dict(a=a, b=b, g=g)
    raise KeyError(name)


def small_dims(name: str) -> dict:
    """Sizes with the same structure as the workload, small enough for the full
    oracle in well under a second, spanning several tiles plus ragged tails."""
    return {
        "c1": dict(P=5, M=67, Q=131),
        "c2": dict(R=333, C=1030),
        "c3": dict(B=3, T=97, C=772),
        "c4": dict(N=2, H=3, T=131),
        "c5a": dict(P=5, M=67, Q=203),
        "c5b": dict(a=(3, 1, 5, 1, 4, 1, 7, 12), b=(1, 2, 1, 3, 1, 5, 1, 12)),
        "x1": dict(R=333, C=1030),
        "u1": dict(R=97, C=1031),
        "c4h": dict(N=2, H=3, T=132),
        "u1h": dict(R=97, C=1032),
        "c3f": dict(B=3, T=97, C=772),
        # 132 columns: 16-byte vectors, so the fused one-pass backward runs.
        "c4f": dict(N=2, H=3, T=132),
    }[name]
