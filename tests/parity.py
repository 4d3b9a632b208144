"""Helpers shared by the GPU parity tests: run a workload's op steps through
the CUDA library and through the CPU oracle on the same seeded host inputs,
and compare.

Acceptance (the operators' contract):
* forward outputs, and gradients that are one exact IEEE operation of their
  inputs (add/sub copy or negation, mul g*b / g*a, div g/b when nothing is
  summed), must be bit-identical, any NaN matching any NaN;
* every summed gradient, and div's -g*a/b^2, must be within
  1e-5 * sum|terms| of the oracle's binary64 result, per element.
"""
from __future__ import annotations

import numpy as np
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads

TOL = 1e-5


def bitexact(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    gn, rn = np.isnan(gpu), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    gb, rb = gpu.view(np.uint32)[~gn], ref.view(np.uint32)[~rn]
    bad = np.nonzero(gb != rb)[0]
    assert bad.size == 0, (f"{what}: {bad.size} elements differ; first at flat {bad[0]}: "
                           f"gpu {gpu[~gn][bad[0]]!r} ref {ref[~rn][bad[0]]!r}")


def within(gpu: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray, what: str = "", tol=TOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    abs_sum = np.asarray(abs_sum, np.float64)
    assert gpu.shape == ref.shape == abs_sum.shape, (what, gpu.shape, ref.shape, abs_sum.shape)
    gn, rn = np.isnan(gpu), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    fin = ~gn & np.isfinite(ref) & np.isfinite(abs_sum)
    inf = ~gn & ~fin
    assert np.array_equal(gpu[inf], ref[inf]) or not inf.any(), f"{what}: infinities differ"
    err = np.abs(gpu[fin] - ref[fin])
    bound = tol * abs_sum[fin]
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} elements beyond {tol}*sum|terms|; worst ratio "
                           f"{np.max(err / np.maximum(bound, 1e-300)):.3g}")


def gelu_close(got, ref, x, mag, what=""):
    """GeLU results against the oracle: within (16 + 2 x^2) * 2^-24 * mag +
    2^-120 per element (mag: |exact| forward; |g| (Phi(x) + |x| phi(x))
    backward), NaN matching NaN and infinities equal.  The x^2 term: binary32
    rounding of the argument x / sqrt(2) (and of the constant 1/sqrt(2)) moves
    erfc(z) far in its tail by a relative z^2 * 2u each, z^2 = x^2 / 2."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    x = np.asarray(x, np.float64)
    mag = np.asarray(mag, np.float64)
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ"
    fin = ~gn & np.isfinite(ref)
    assert np.array_equal(got[~gn & ~fin], ref[~gn & ~fin]), f"{what}: infinities differ"
    bound = (16.0 + 2.0 * x[fin] ** 2) * 2.0 ** -24 * mag[fin] + 2.0 ** -120
    err = np.abs(got[fin] - ref[fin])
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} beyond bound; worst at x={x[fin][bad[0]]}: "
                           f"gpu {got[fin][bad[0]]} ref {ref[fin][bad[0]]}")


def is_single_op_grad(op: str, which: int, reduced: bool) -> bool:
    """True if a gradient element is exactly one IEEE op of the inputs."""
    if reduced:
        return False
    return not (op == "div" and which == 1)


def to_gpu(x: torch.Tensor) -> torch.Tensor:
    """Device copy with the same strides and storage offset: the whole
    underlying storage is copied and the view rebuilt over it, so transposed,
    stepped and misaligned views keep their layout on the GPU."""
    st = x.untyped_storage()
    n = st.nbytes() // x.element_size()
    flat = torch.empty(0, dtype=x.dtype).set_(st, 0, (n,), (1,))
    dev = flat.cuda()
    return dev.as_strided(x.shape, x.stride(), x.storage_offset())


def run_gpu(name: str, host: dict) -> dict:
    """All step outputs of workload ``name`` computed by the CUDA library."""
    env = {k: to_gpu(v) for k, v in host.items()}
    for step in workloads.STEPS[name]:
        if step[0] == "ufwd":
            _, op, alpha, xn, on = step
            env[on] = zr.zr_unary_fwd(op, env[xn], alpha=alpha)
        elif step[0] == "ubwd":
            _, op, alpha, gn, xn, gxn = step
            env[gxn] = zr.zr_unary_bwd(op, env[gn], env[xn], alpha=alpha)
        elif step[0] == "cfwd":
            _, op1, op2, an, bn, cn, on = step
            env[on] = zr.zr_chain_fwd(op1, op2, env[an], env[bn], env[cn])
        elif step[0] == "cbwd":
            _, op1, op2, gn, an, bn, cn, gan, gbn, gcn = step
            env[gan], env[gbn], env[gcn] = zr.zr_chain_bwd(op1, op2, env[gn], env[an], env[bn],
                                                           env[cn])
        elif step[0] == "fwd":
            _, op, an, bn, on = step
            env[on] = zr.zr_binary_fwd(op, env[an], env[bn])
        else:
            _, op, gn, an, bn, gan, gbn = step
            ga, gb = zr.zr_binary_bwd(op, env[gn], env[an], env[bn])
            env[gan], env[gbn] = ga, gb
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in env.items()}


def run_oracle(name: str, host: dict) -> tuple[dict, dict]:
    """(values, abs_sums) of every step output, computed by the oracle."""
    env = {k: v for k, v in host.items()}
    sums = {}
    for step in workloads.STEPS[name]:
        if step[0] == "ufwd":
            _, op, alpha, xn, on = step
            env[on] = torch.from_numpy(oracle.unary_fwd(op, env[xn], alpha=alpha))
            sums[on] = np.abs(env[on].numpy().astype(np.float64))
        elif step[0] == "ubwd":
            _, op, alpha, gn, xn, gxn = step
            r, mag = oracle.unary_bwd(op, env[gn], env[xn], alpha=alpha)
            env[gxn] = torch.from_numpy(r)
            sums[gxn] = mag
        elif step[0] == "cfwd":
            _, op1, op2, an, bn, cn, on = step
            env[on] = torch.from_numpy(oracle.chain_fwd(op1, op2, env[an], env[bn], env[cn]))
        elif step[0] == "cbwd":
            _, op1, op2, gn, an, bn, cn, gan, gbn, gcn = step
            r = oracle.chain_bwd(op1, op2, env[gn], env[an], env[bn], env[cn])
            for k, nm in enumerate((gan, gbn, gcn)):
                env[nm] = torch.from_numpy(r[k])
                sums[nm] = r[3 + k]
        elif step[0] == "fwd":
            _, op, an, bn, on = step
            env[on] = torch.from_numpy(oracle.binary_fwd(op, env[an], env[bn]))
        else:
            _, op, gn, an, bn, gan, gbn = step
            ga, gb, sa, sb = oracle.binary_bwd(op, env[gn], env[an], env[bn])
            env[gan], env[gbn] = torch.from_numpy(ga), torch.from_numpy(gb)
            sums[gan], sums[gbn] = sa, sb
    return env, sums


def compare_workload(name: str, host: dict, gpu: dict, ref: dict, sums: dict):
    out_shapes = {}
    for step in workloads.STEPS[name]:
        if step[0] in ("ufwd", "ubwd"):
            op, xn, on = step[1], step[-2], step[-1]
            what = f"{name} {step[0]} {op} -> {on}"
            if op == "scale":
                bitexact(gpu[on].numpy(), ref[on].numpy(), what)
            else:
                gelu_close(gpu[on].numpy(), ref[on].numpy(), host[xn].numpy(), sums[on], what)
            continue
        if step[0] == "cfwd":
            on = step[6]
            bitexact(gpu[on].numpy(), ref[on].numpy(), f"{name} chain fwd -> {on}")
            continue
        if step[0] == "cbwd":
            _, op1, op2, gn, an, bn, cn, gan, gbn, gcn = step
            n_out = ref[gn].numel()
            t_full = int(np.prod(np.broadcast_shapes(tuple(ref[an].shape), tuple(ref[bn].shape)))) == n_out
            for k, (src, gname) in enumerate(((an, gan), (bn, gbn), (cn, gcn))):
                full = ref[gname].numel() == n_out
                exact = full and ((k == 0 and t_full) or (k == 1 and t_full and op1 != "div") or
                                  (k == 2 and op2 != "div"))
                what = f"{name} chain bwd -> {gname}"
                if exact:
                    bitexact(gpu[gname].numpy(), ref[gname].numpy(), what)
                else:
                    within(gpu[gname].numpy(), ref[gname].numpy(), sums[gname], what)
            continue
        if step[0] == "fwd":
            _, op, an, bn, on = step
            bitexact(gpu[on].numpy(), ref[on].numpy(), f"{name} fwd {op} -> {on}")
            out_shapes[on] = tuple(ref[on].shape)
        else:
            _, op, gn, an, bn, gan, gbn = step
            out_numel = ref[gn].numel()
            for which, gname, src in ((0, gan, an), (1, gbn, bn)):
                reduced = ref[gname].numel() != out_numel
                what = f"{name} bwd {op} -> {gname}"
                if is_single_op_grad(op, which, reduced):
                    bitexact(gpu[gname].numpy(), ref[gname].numpy(), what)
                else:
                    within(gpu[gname].numpy(), ref[gname].numpy(), sums[gname], what)
