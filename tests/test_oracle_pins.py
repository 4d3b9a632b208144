"""Pins of the CPU oracle to facts outside itself (CPU only, no GPU).

Each test checks the oracle against something the pages print, a library
routine that implements the same rule (NumPy broadcasting and binary32
arithmetic), a closed form, float64 finite differences, or a second
formulation of the same definition.  Chosen so that a dropped term, a flipped
sign, a wrong index or a transposed operand in the oracle fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
OPS = ["add", "sub", "mul", "div"]
NP_OP = {"add": np.add, "sub": np.subtract, "mul": np.multiply, "div": np.divide}


def _ints(s):
    s = s.strip()
    return tuple(int(v) for v in s.split(",")) if s else ()


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- broadcast shape

def test_broadcast_printed_examples():
    for ln in _golden_lines("broadcast_examples.txt"):
        sa, sb, res = (p.strip() for p in ln.split(";"))
        if res == "reject":
            with pytest.raises(oracle.OracleError):
                oracle.broadcast_shape(_ints(sa), _ints(sb))
        else:
            assert oracle.broadcast_shape(_ints(sa), _ints(sb)) == _ints(res)


def _rand_pair(rng, max_nd=8, allow_zero=True):
    na, nb = rng.integers(0, max_nd + 1, size=2)
    n = max(na, nb)
    base = rng.integers(0 if allow_zero else 1, 5, size=n)
    sa = [int(v) if rng.random() < 0.6 else 1 for v in base[n - na:]]
    sb = [int(v) if rng.random() < 0.6 else 1 for v in base[n - nb:]]
    if rng.random() < 0.2 and nb > 0:  # sometimes incompatible
        sb[rng.integers(0, nb)] = int(rng.integers(2, 7))
    return sa, sb


def test_broadcast_matches_numpy_and_is_symmetric():
    rng = np.random.default_rng(7)
    n_ok = n_bad = 0
    for _ in range(3000):
        sa, sb = _rand_pair(rng)
        try:
            ref = tuple(np.broadcast_shapes(tuple(sa), tuple(sb)))
        except ValueError:
            ref = None
        if ref is None:
            n_bad += 1
            with pytest.raises(oracle.OracleError):
                oracle.broadcast_shape(sa, sb)
            with pytest.raises(oracle.OracleError):
                oracle.broadcast_shape(sb, sa)
        else:
            n_ok += 1
            assert oracle.broadcast_shape(sa, sb) == ref
            assert oracle.broadcast_shape(sb, sa) == ref
    assert n_ok > 500 and n_bad > 100


def test_broadcast_rank_limit():
    with pytest.raises(oracle.OracleError):
        oracle.broadcast_shape([1] * 9, [1])


# ---------------------------------------------------------------- strides and index map

def test_stride_printed_examples():
    lines = _golden_lines("stride_examples.txt")
    storage = np.array(_ints(lines[0].split(":", 1)[1]), dtype=np.float32)
    n_read = 0
    for ln in lines[1:]:
        kind, rest = ln.split(":", 1)
        if kind == "strides":
            shape, strides = (p.strip() for p in rest.split("->"))
            assert oracle.contiguous_strides(_ints(shape)) == _ints(strides)
        elif kind == "read":
            lhs, val = rest.split("->")
            sizes, strides, coord = (_ints(p) for p in lhs.split(";"))
            view = np.lib.stride_tricks.as_strided(
                storage, shape=sizes, strides=tuple(4 * s for s in strides))
            # Read through the oracle's strided index map: add +0.0 (exact).
            out = oracle.binary_fwd("add", view, np.zeros((1,), np.float32))
            assert out[coord] == float(val)
            n_read += 1
    assert n_read == 2


def test_contiguous_strides_match_numpy():
    rng = np.random.default_rng(3)
    for _ in range(200):
        shape = tuple(int(v) for v in rng.integers(1, 6, size=rng.integers(0, 9)))
        ref = tuple(s // 4 for s in np.empty(shape, np.float32).strides)
        assert oracle.contiguous_strides(shape) == ref


def test_broadcast_rows_printed_example():
    (ln,) = _golden_lines("broadcast_rows.txt")
    vals, shape, target, rows = (p.strip() for p in ln.split(";"))
    x = np.array(_ints(vals), np.float32).reshape(_ints(shape))
    out = oracle.binary_fwd("add", np.zeros(_ints(target), np.float32), x)
    expect = np.array([_ints(r) for r in rows.split("|")], np.float32)
    np.testing.assert_array_equal(out, expect)


# ---------------------------------------------------------------- forward

def _strided(rng, shape):
    """A float32 view of ``shape`` with non-trivial strides (permuted storage,
    stepped slices or expanded size-1 dims), plus its dense copy."""
    kind = rng.integers(0, 3)
    if kind == 0 or len(shape) < 2:
        x = rng.standard_normal(shape).astype(np.float32)
        return x
    if kind == 1:
        perm = rng.permutation(len(shape))
        base = rng.standard_normal(tuple(shape[p] for p in perm)).astype(np.float32)
        return np.transpose(base, np.argsort(perm))
    big = rng.standard_normal(tuple(2 * s for s in shape)).astype(np.float32)
    return big[tuple(slice(0, 2 * s, 2) for s in shape)]


def test_forward_matches_numpy_float32_bit_exact():
    rng = np.random.default_rng(11)
    for it in range(400):
        sa, sb = _rand_pair(rng, max_nd=5, allow_zero=True)
        try:
            ref_shape = np.broadcast_shapes(tuple(sa), tuple(sb))
        except ValueError:
            continue
        a = _strided(rng, tuple(sa))
        b = _strided(rng, tuple(sb))
        if rng.random() < 0.3:
            b = np.where(rng.random(b.shape) < 0.3, np.float32(0.0), b).astype(np.float32)
        op = OPS[it % 4]
        out = oracle.binary_fwd(op, a, b)
        with np.errstate(all="ignore"):
            ref = NP_OP[op](a, b).astype(np.float32)
        assert out.shape == tuple(ref_shape)
        np.testing.assert_array_equal(out.view(np.uint32)[~np.isnan(ref)],
                                      ref.view(np.uint32)[~np.isnan(ref)])
        assert np.array_equal(np.isnan(out), np.isnan(ref))


def test_forward_special_values_bit_exact():
    sp = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45,
                   1.17e-38, 3.4e38, -3.4e38, 8.0, 0.125, 1e-30], np.float32)
    a = sp.reshape(-1, 1)
    b = sp.reshape(1, -1)
    for op in OPS:
        out = oracle.binary_fwd(op, a, b)
        with np.errstate(all="ignore"):
            ref = NP_OP[op](a, b)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(out), nan)
        np.testing.assert_array_equal(out.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def test_forward_division_by_power_of_two_is_exact_scaling():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(4096) * 1e3).astype(np.float32)
    out = oracle.binary_fwd("div", a, np.array([8.0], np.float32))
    np.testing.assert_array_equal(out, a * np.float32(0.125))


def test_forward_at_matches_full():
    x = workloads.make_inputs("c5b", **workloads.small_dims("c5b"))
    full = oracle.binary_fwd("div", x["a"], x["b"]).reshape(-1)
    idx = np.random.default_rng(0).integers(0, full.size, 500)
    np.testing.assert_array_equal(oracle.binary_fwd_at("div", x["a"], x["b"], idx), full[idx])


# ---------------------------------------------------------------- backward

def test_worked_gradient_example():
    kv = {}
    for ln in _golden_lines("worked_gradient.txt"):
        k, v = (p.strip() for p in ln.split("="))
        kv[k] = float(v)
    x = np.array([kv["x"]], np.float32)
    y = np.array([kv["y"]], np.float32)
    xy = oracle.binary_fwd("mul", x, y)
    z = oracle.binary_fwd("add", xy, x)
    assert xy[0] == kv["xy"] and z[0] == kv["z"]
    one = np.ones(1, np.float32)
    g_xy, g_x_add, _, _ = oracle.binary_bwd("add", one, xy, x)
    g_x_mul, g_y, _, _ = oracle.binary_bwd("mul", g_xy, x, y)
    # The caller accumulates x's two paths.
    assert g_x_mul[0] + g_x_add[0] == kv["dz_dx"]
    assert g_y[0] == kv["dz_dy"]


def _loss64(op, a64, b64, w64):
    with np.errstate(all="ignore"):
        return float(np.sum(w64 * NP_OP[op](a64, b64)))


@pytest.mark.parametrize("op", OPS)
def test_backward_matches_finite_differences(op):
    rng = np.random.default_rng(100 + OPS.index(op))
    shapes = [((3, 4), (4,)), ((2, 1, 3), (4, 1)), ((1, 5), (3, 1)), ((2, 3), (2, 3)),
              ((4,), (1,)), ((2, 1, 3, 1), (1, 2, 1, 2))]
    for sa, sb in shapes:
        a = rng.standard_normal(sa).astype(np.float32)
        b = rng.standard_normal(sb).astype(np.float32)
        if op == "div":
            b = (np.sign(b) * (0.5 + np.abs(b))).astype(np.float32)
        out_shape = np.broadcast_shapes(sa, sb)
        w = rng.standard_normal(out_shape).astype(np.float32)
        ga, gb, _, _ = oracle.binary_bwd(op, w, a, b)
        a64, b64, w64 = a.astype(np.float64), b.astype(np.float64), w.astype(np.float64)
        for x64, grad in ((a64, ga), (b64, gb)):
            fd = np.empty(x64.shape)
            for i in np.ndindex(x64.shape):
                h = 1e-6 * max(1.0, abs(x64[i]))
                keep = x64[i]
                x64[i] = keep + h
                lp = _loss64(op, a64, b64, w64)
                x64[i] = keep - h
                lm = _loss64(op, a64, b64, w64)
                x64[i] = keep
                fd[i] = (lp - lm) / (2 * h)
            np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("op", OPS)
def test_backward_matches_numpy_reduction(op):
    """Gradient = NumPy float64 sum, over the broadcast axes, of the local
    terms; independent of the oracle's index bookkeeping."""
    rng = np.random.default_rng(200 + OPS.index(op))
    for sa, sb in [((5, 1, 7), (3, 1)), ((2, 3, 1, 4), (1, 3, 5, 1)), ((6,), (2, 1, 6))]:
        a = _strided(rng, sa)
        b = (np.sign(rng.standard_normal(sb)) * (0.5 + rng.random(sb))).astype(np.float32)
        out_shape = np.broadcast_shapes(sa, sb)
        g = rng.standard_normal(out_shape).astype(np.float32)
        ga, gb, _, _ = oracle.binary_bwd(op, g, a, b)
        A = np.broadcast_to(a.astype(np.float64), out_shape)
        B = np.broadcast_to(b.astype(np.float64), out_shape)
        G = g.astype(np.float64)
        ta = {"add": G, "sub": G, "mul": G * B, "div": G / B}[op]
        tb = {"add": G, "sub": -G, "mul": G * A, "div": -(G * A) / (B * B)}[op]

        def reduce_to(t, shape):
            lead = len(out_shape) - len(shape)
            axes = tuple(range(lead)) + tuple(
                lead + i for i, s in enumerate(shape) if s == 1 and out_shape[lead + i] != 1)
            return np.sum(t, axis=axes).reshape(shape)

        ra, rb = reduce_to(ta, sa), reduce_to(tb, sb)
        np.testing.assert_allclose(ga, ra.astype(np.float32), rtol=2 ** -23, atol=1e-30)
        np.testing.assert_allclose(gb, rb.astype(np.float32), rtol=2 ** -23, atol=1e-30)


def test_single_term_gradients_are_the_fp32_op_bit_exact():
    rng = np.random.default_rng(9)
    a = rng.standard_normal((64, 33)).astype(np.float32)
    b = (rng.standard_normal((64, 33)) + 3).astype(np.float32)
    g = rng.standard_normal((64, 33)).astype(np.float32)
    g[0, :5] = [0.0, -0.0, np.inf, 1e-45, -3.0]
    ga, gb, _, _ = oracle.binary_bwd("mul", g, a, b)
    np.testing.assert_array_equal(ga.view(np.uint32), (g * b).view(np.uint32))
    np.testing.assert_array_equal(gb.view(np.uint32), (g * a).view(np.uint32))
    ga, _, _, _ = oracle.binary_bwd("div", g, a, b, want_b=False)
    np.testing.assert_array_equal(ga.view(np.uint32), (g / b).view(np.uint32))
    ga, gb, _, _ = oracle.binary_bwd("sub", g, None, None, shape_a=g.shape, shape_b=g.shape)
    np.testing.assert_array_equal(ga.view(np.uint32), g.view(np.uint32))
    np.testing.assert_array_equal(gb.view(np.uint32), (-g).view(np.uint32))


def test_backward_invariants():
    rng = np.random.default_rng(12)
    g = rng.standard_normal((6, 5, 7)).astype(np.float32)
    ga_add, gb_add, sa, sb = oracle.binary_bwd("add", g, None, None,
                                               shape_a=(6, 5, 7), shape_b=(5, 1))
    total = math.fsum(g.astype(np.float64).ravel())
    assert abs(math.fsum(ga_add.astype(np.float64).ravel()) - total) <= 1e-5 * np.abs(g).sum()
    assert abs(math.fsum(gb_add.astype(np.float64).ravel()) - total) <= 1e-5 * np.abs(g).sum()
    _, gb_sub, _, _ = oracle.binary_bwd("sub", g, None, None, shape_a=(6, 5, 7), shape_b=(5, 1))
    np.testing.assert_array_equal(gb_sub.view(np.uint32), (-gb_add).view(np.uint32))
    a = rng.standard_normal((6, 5, 7)).astype(np.float32)
    ga_mul, _, _, _ = oracle.binary_bwd("mul", g, a, np.ones((5, 1), np.float32))
    np.testing.assert_array_equal(ga_mul.view(np.uint32), g.view(np.uint32))
    np.testing.assert_allclose(sb.ravel(), np.abs(g.astype(np.float64)).sum(axis=(0, 2)))


@pytest.mark.parametrize("name", ["c1", "c5a", "c5b"])
def test_scatter_and_gather_backward_agree(name):
    x = workloads.make_inputs(name, **workloads.small_dims(name))
    step = workloads.STEPS[name][-1]
    _, op, gn, an, bn, _, _ = step
    g, a, b = x[gn], x[an], x[bn]
    ga, gb, sa, sb = oracle.binary_bwd(op, g, a, b)
    rng = np.random.default_rng(1)
    for which, full, fabs in ((0, ga, sa), (1, gb, sb)):
        idx = rng.integers(0, full.size, 300)
        v, s = oracle.binary_bwd_at(op, which, g, a, b, idx)
        np.testing.assert_array_equal(v, full.reshape(-1)[idx])
        np.testing.assert_array_equal(s, fabs.reshape(-1)[idx])


# ---------------------------------------------------------------- sum to shape

def test_sum_to_shape_closed_forms():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((9, 11, 13)).astype(np.float32)
    same, _ = oracle.sum_to_shape(x, x.shape)
    np.testing.assert_array_equal(same.view(np.uint32), x.view(np.uint32))
    one, sabs = oracle.sum_to_shape(x, (1,))
    exact = math.fsum(x.astype(np.float64).ravel())
    assert abs(float(one[0]) - exact) <= 2 ** -24 * abs(exact) + 1e-30
    assert abs(sabs[0] - math.fsum(np.abs(x.astype(np.float64)).ravel())) <= 1e-9
    col, _ = oracle.sum_to_shape(x.reshape(99, 13), (13,))
    for c in range(13):
        e = math.fsum(x.reshape(99, 13)[:, c].astype(np.float64))
        assert abs(float(col[c]) - e) <= 2 ** -24 * abs(e) + 1e-30
    mid, _ = oracle.sum_to_shape(x, (11, 1))
    for m in range(11):
        e = math.fsum(x[:, m, :].astype(np.float64).ravel())
        assert abs(float(mid[m, 0]) - e) <= 2 ** -24 * abs(e) + 1e-30


def test_sum_to_shape_strided_and_gather_agree():
    t = torch.randn(7, 5, 9, generator=torch.Generator().manual_seed(4)).permute(2, 0, 1)
    full, fabs = oracle.sum_to_shape(t, (9, 1, 5))
    ref = t.double().sum(dim=1, keepdim=True)
    np.testing.assert_allclose(full, ref.float().numpy(), rtol=2 ** -23, atol=0)
    idx = np.arange(full.size)
    v, s = oracle.sum_to_shape_at(t, (9, 1, 5), idx)
    np.testing.assert_array_equal(v, full.reshape(-1))
    np.testing.assert_array_equal(s, fabs.reshape(-1))


def test_sum_to_shape_rejects_non_broadcast_target():
    x = np.zeros((4, 6), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.sum_to_shape(x, (4, 3))
    with pytest.raises(oracle.OracleError):
        oracle.sum_to_shape(x, (2, 4, 6))


def test_empty_shapes():
    a = np.zeros((0, 3), np.float32)
    b = np.ones((1, 3), np.float32)
    assert oracle.binary_fwd("add", a, b).shape == (0, 3)
    ga, gb, _, _ = oracle.binary_bwd("mul", np.zeros((0, 3), np.float32), a, b)
    assert ga.shape == (0, 3)
    np.testing.assert_array_equal(gb, np.zeros((1, 3), np.float32))


# ---------------------------------------------------------------- two-op chains

def test_chain_worked_gradient_example():
    """z = x*y + x is the chain (x mul y) add x: the book's worked example."""
    kv = {}
    for ln in _golden_lines("worked_gradient.txt"):
        k, v = (p.strip() for p in ln.split("="))
        kv[k] = float(v)
    x = np.array([kv["x"]], np.float32)
    y = np.array([kv["y"]], np.float32)
    z = oracle.chain_fwd("mul", "add", x, y, x)
    assert z[0] == kv["z"]
    ga, gb, gc, _, _, _ = oracle.chain_bwd("mul", "add", np.ones(1, np.float32), x, y, x)
    # x enters twice (as a and as c); the caller adds its two gradients.
    assert ga[0] + gc[0] == kv["dz_dx"]
    assert gb[0] == kv["dz_dy"]


CHAIN_SHAPES = [((3, 4), (4,), (3, 1)), ((2, 1, 3), (4, 1), (3,)), ((2, 3), (2, 3), (1,)),
                ((4,), (1,), (2, 4)), ((2, 3, 4), (3, 1), (2, 1, 4))]


def _chain_inputs(rng, sa, sb, sc, op1, op2):
    a = rng.standard_normal(sa).astype(np.float32)
    b = rng.standard_normal(sb).astype(np.float32)
    c = rng.standard_normal(sc).astype(np.float32)
    if op1 == "div":
        b = (np.sign(b) * (0.5 + np.abs(b))).astype(np.float32)
    if op2 == "div":
        c = (np.sign(c) * (0.5 + np.abs(c))).astype(np.float32)
    return a, b, c


@pytest.mark.parametrize("op1", OPS)
def test_chain_forward_matches_numpy_float32_bit_exact(op1):
    rng = np.random.default_rng(500 + OPS.index(op1))
    for op2 in OPS:
        for sa, sb, sc in CHAIN_SHAPES:
            a, b, c = _chain_inputs(rng, sa, sb, sc, op1, op2)
            with np.errstate(all="ignore"):
                ref = NP_OP[op2](NP_OP[op1](a, b), c).astype(np.float32)
            got = oracle.chain_fwd(op1, op2, a, b, c)
            assert got.shape == ref.shape
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (op1, op2, sa, sb, sc)


def _chain_loss64(op1, op2, a64, b64, c64, w64):
    with np.errstate(all="ignore"):
        return float(np.sum(w64 * NP_OP[op2](NP_OP[op1](a64, b64), c64)))


@pytest.mark.parametrize("op1", OPS)
def test_chain_backward_matches_finite_differences(op1):
    rng = np.random.default_rng(600 + OPS.index(op1))
    for op2 in OPS:
        for sa, sb, sc in CHAIN_SHAPES:
            a, b, c = _chain_inputs(rng, sa, sb, sc, op1, op2)
            out_shape = np.broadcast_shapes(sa, sb, sc)
            w = rng.standard_normal(out_shape).astype(np.float32)
            grads = oracle.chain_bwd(op1, op2, w, a, b, c)[:3]
            xs = [a.astype(np.float64), b.astype(np.float64), c.astype(np.float64)]
            w64 = w.astype(np.float64)
            for k in range(3):
                x64, grad = xs[k], grads[k]
                fd = np.empty(x64.shape)
                for i in np.ndindex(x64.shape):
                    h = 1e-6 * max(1.0, abs(x64[i]))
                    keep = x64[i]
                    x64[i] = keep + h
                    lp = _chain_loss64(op1, op2, *xs, w64)
                    x64[i] = keep - h
                    lm = _chain_loss64(op1, op2, *xs, w64)
                    x64[i] = keep
                    fd[i] = (lp - lm) / (2 * h)
                np.testing.assert_allclose(grad, fd, rtol=2e-5, atol=2e-5,
                                           err_msg=f"{op1} {op2} {sa} {sb} {sc} input {k}")


def test_chain_affine_closed_form():
    """(x * gamma) + beta: grad_x = g*gamma (one binary32 multiply),
    grad_gamma = column sums of g*x, grad_beta = column sums of g."""
    host = workloads.make_inputs("c3", **workloads.small_dims("c3"))
    x, gamma, beta, g = (host[k].numpy() for k in ("x", "gamma", "beta", "g"))
    ga, gb, gc, sa, sb, sc = oracle.chain_bwd("mul", "add", g, x, gamma, beta)
    ref_x = (g * gamma).astype(np.float32)
    assert np.array_equal(ga.view(np.uint32), ref_x.view(np.uint32))
    g64, x64 = g.astype(np.float64), x.astype(np.float64)
    col_gx = np.sum(g64 * x64, axis=(0, 1))
    col_g = np.sum(g64, axis=(0, 1))
    assert np.all(np.abs(gb - col_gx) <= 1e-6 * np.sum(np.abs(g64 * x64), axis=(0, 1)))
    assert np.all(np.abs(gc - col_g) <= 1e-6 * np.sum(np.abs(g64), axis=(0, 1)))
    np.testing.assert_allclose(sb, np.sum(np.abs(g64 * x64), axis=(0, 1)), rtol=1e-6)


def test_chain_scaled_mask_closed_form():
    """(scores + mask) / k: grad_scores = g/k (one binary32 division),
    grad_mask = sums of g/k over batch and heads, grad_k = -sum(g*t)/k^2
    with t = fl32(scores + mask)."""
    host = workloads.make_inputs("c4", **workloads.small_dims("c4"))
    s, m, k, g = (host[n].numpy() for n in ("scores", "mask", "scalar", "g"))
    ga, gb, gc, sa, sb, sc = oracle.chain_bwd("add", "div", g, s, m, k)
    assert np.array_equal(ga.view(np.uint32), (g / k).astype(np.float32).view(np.uint32))
    g64 = g.astype(np.float64)
    k64 = float(k[0])
    mask_ref = np.sum(g64 / k64, axis=(0, 1), keepdims=True)
    assert np.all(np.abs(gb - mask_ref) <= 1e-6 * np.sum(np.abs(g64 / k64), axis=(0, 1), keepdims=True))
    t64 = (s + m).astype(np.float32).astype(np.float64)
    terms = -g64 * t64 / (k64 * k64)
    assert abs(float(gc[0]) - math.fsum(terms.ravel())) <= 1e-6 * float(np.sum(np.abs(terms)))


def test_chain_gather_form_matches_full():
    rng = np.random.default_rng(700)
    for op1, op2 in (("mul", "add"), ("add", "div"), ("div", "mul"), ("sub", "sub")):
        for sa, sb, sc in CHAIN_SHAPES:
            a, b, c = _chain_inputs(rng, sa, sb, sc, op1, op2)
            g = rng.standard_normal(np.broadcast_shapes(sa, sb, sc)).astype(np.float32)
            full = oracle.chain_bwd(op1, op2, g, a, b, c)
            for which, shape in enumerate((sa, sb, sc)):
                idx = np.arange(int(np.prod(shape)), dtype=np.int64)
                vals, sabs = oracle.chain_bwd_at(op1, op2, which, g, a, b, c, idx)
                assert np.array_equal(vals.view(np.uint32), full[which].ravel().view(np.uint32))
                np.testing.assert_allclose(sabs, full[3 + which].ravel(), rtol=1e-12)


def test_accumulate_worked_gradient_example():
    """x reaches z = x*y + x along two paths; the book adds their gradients
    into x's slot: 2 (through Mul) + 1 (through Add) = dz/dx = 3."""
    kv = {}
    for ln in _golden_lines("worked_gradient.txt"):
        k, v = (p.strip() for p in ln.split("="))
        kv[k] = float(v)
    x = np.array([kv["x"]], np.float32)
    y = np.array([kv["y"]], np.float32)
    xy = oracle.binary_fwd("mul", x, y)
    one = np.ones(1, np.float32)
    g_xy, g_x_add, _, _ = oracle.binary_bwd("add", one, xy, x)
    g_x_mul, _, _, _ = oracle.binary_bwd("mul", g_xy, x, y)
    slot = np.zeros(1, np.float32)
    slot = oracle.accumulate(slot, g_x_mul)
    slot = oracle.accumulate(slot, g_x_add)
    assert slot[0] == kv["dz_dx"]


def test_accumulate_is_one_rounded_addition():
    """Each element is old + new rounded once: by Figueroa's double-rounding
    result a binary64 sum of two binary32 values rounded to binary32 is that
    value; the sign rules of zero follow IEEE (+0 + -0 = +0)."""
    rng = np.random.default_rng(21)
    old = (rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000)).astype(np.float32)
    new = (rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000)).astype(np.float32)
    got = oracle.accumulate(old, new)
    want = (old.astype(np.float64) + new.astype(np.float64)).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    z = oracle.accumulate(np.array([0.0, -0.0, -0.0], np.float32), np.array([-0.0, 0.0, -0.0], np.float32))
    assert list(np.signbit(z)) == [False, False, True]


# ---------------------------------------------------------------- unary ops

def test_unary_scale_is_one_float32_multiply():
    rng = np.random.default_rng(31)
    base = torch.from_numpy(rng.standard_normal((40, 30)).astype(np.float32))
    x = base.t()  # strided view
    for alpha in (0.125, -3.0, 1e-30, 7.5):
        got = oracle.unary_fwd("scale", x, alpha=alpha)
        want = (np.float32(alpha) * x.numpy()).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
        g = rng.standard_normal((30, 40)).astype(np.float32)
        gx, mag = oracle.unary_bwd("scale", g, None, alpha=alpha)
        assert np.array_equal(gx.view(np.uint32), (np.float32(alpha) * g).astype(np.float32).view(np.uint32))


def test_gelu_printed_normal_cdf_values():
    for ln in _golden_lines("normal_cdf.txt"):
        xs, ps = (p.strip() for p in ln.split(";"))
        x, phi = float(xs), float(ps)
        got = float(oracle.unary_fwd("gelu", np.array([x], np.float32))[0])
        assert abs(got - x * phi) <= 2.0 ** -24 * abs(x * phi) + 1e-10, (x, got, x * phi)
    # GeLU'(0) = Phi(0) = 1/2 exactly.
    gx, _ = oracle.unary_bwd("gelu", np.ones(1, np.float32), np.zeros(1, np.float32))
    assert gx[0] == 0.5


def test_gelu_odd_identity_and_erf_form():
    """x Phi(x) - (-x) Phi(-x) = x; and the erf form 0.5 x (1 + erf(x/sqrt 2))
    (a different library function) agrees where it does not cancel."""
    rng = np.random.default_rng(32)
    x = (rng.standard_normal(4000) * 3).astype(np.float32)
    p, m = oracle.unary_fwd("gelu", x), oracle.unary_fwd("gelu", -x)
    err = np.abs((p.astype(np.float64) - m.astype(np.float64)) - x.astype(np.float64))
    assert np.all(err <= 2.0 ** -23 * (np.abs(p) + np.abs(m)) + 1e-30)
    xs = x[np.abs(x) <= 3.0]
    ref = np.array([0.5 * float(v) * (1.0 + math.erf(float(v) / math.sqrt(2.0))) for v in xs])
    got = oracle.unary_fwd("gelu", xs).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -23 * np.abs(ref) + 1e-12)


def test_gelu_backward_matches_finite_differences():
    rng = np.random.default_rng(33)
    x = (rng.standard_normal(300) * 2).astype(np.float32)
    g = rng.standard_normal(300).astype(np.float32)
    gx, mag = oracle.unary_bwd("gelu", g, x)

    def f(v):
        return 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))
    for i in range(x.size):
        v = float(x[i])
        h = 1e-6 * max(1.0, abs(v))
        fd = float(g[i]) * (f(v + h) - f(v - h)) / (2 * h)
        assert abs(float(gx[i]) - fd) <= 1e-6 * float(mag[i]) + 1e-7, (v, gx[i], fd)
        assert abs(float(gx[i])) <= float(mag[i]) * (1 + 1e-6)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_conversion():
    """The oracle's bf16 rounding against PyTorch's float32 -> bfloat16
    conversion (round to nearest, ties to even), including ties, overflow to
    infinity, subnormals, signed zeros, infinities and NaN."""
    rng = np.random.default_rng(71)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00000001, 0x00008000,
                        0x3F808000, 0x3F818000, 0x7F7F8000], np.uint32)
    for b in (bits, ties, special):
        x = b.view(np.float32)
        got = oracle.round_bf16(x)
        want = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float32).numpy()
        gn, wn = np.isnan(got), np.isnan(want)
        assert np.array_equal(gn, wn)
        assert np.array_equal(got[~gn].view(np.uint32), want[~wn].view(np.uint32))


def test_bf16_single_ops_round_once():
    """bf16 inputs, one binary32 operation, rounded to bf16: equal to the
    exact (binary64) result rounded to bf16 through binary32 (innocuous
    double rounding, 24 >= 2*8+2)."""
    rng = np.random.default_rng(72)
    a = oracle.round_bf16(rng.standard_normal(50000).astype(np.float32) * 3)
    b = oracle.round_bf16((0.5 + rng.random(50000)).astype(np.float32))
    for op in OPS:
        got = oracle.round_bf16(oracle.binary_fwd(op, a, b))
        exact64 = NP_OP[op](a.astype(np.float64), b.astype(np.float64))
        # Round binary64 straight to bf16: nearest representable, ties to even.
        e = np.frexp(exact64)[1]
        step = np.ldexp(1.0, e - 8)
        q = exact64 / step
        r = np.floor(q)
        frac = q - r
        r = np.where((frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1)), r + 1, r)
        want = (r * step).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), op

