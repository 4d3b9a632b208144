"""GPU parity of the two-op chains out = (a op1 b) op2 c (zr_chain_fwd,
zr_chain_bwd) against the CPU oracle's composition of the two binary ops,
through the C ABI.

Acceptance as for the binary ops: the forward, and every gradient that is a
chain of single binary32 operations (grad_a when a has the output's shape;
grad_b / grad_c when they have it and op1 / op2 is not div), bit-identical;
every summed gradient within 1e-5 * sum|terms| of the oracle per element.
Both backward routes are covered: the fused one-pass kernel (a of the output
shape, b reduced, c shaped like b or one element) and the composed route.
"""
import ctypes
import json

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads
from parity import bitexact, to_gpu, within

pytestmark = pytest.mark.gpu

OPS = ["add", "sub", "mul", "div"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    L = zr.lib()
    L.zr_test_describe_chain_bwd.argtypes = [ctypes.c_int, ctypes.c_int, zr.ZrTensor, zr.ZrTensor,
                                             zr.ZrTensor, zr.ZrTensor, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                             ctypes.c_size_t]


def _route(op1, op2, g, a, b, c, grads):
    keep = [zr._desc(x) for x in (g, a, b, c)]
    buf = ctypes.create_string_buffer(8192)
    ptrs = [x.data_ptr() if x is not None else None for x in grads]
    assert zr.lib().zr_test_describe_chain_bwd(zr.OPS[op1], zr.OPS[op2], *[k[0] for k in keep],
                                               *ptrs, buf, 8192) == 0
    return json.loads(buf.value.decode())["route"]


def _nonzero(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    return (np.sign(x) * (0.5 + np.abs(x))).astype(np.float32)


def _inputs(rng, op1, op2, sa, sb, sc):
    a = rng.standard_normal(sa).astype(np.float32)
    b = _nonzero(rng, sb) if op1 == "div" else rng.standard_normal(sb).astype(np.float32)
    c = _nonzero(rng, sc) if op2 == "div" else rng.standard_normal(sc).astype(np.float32)
    g = rng.standard_normal(np.broadcast_shapes(sa, sb, sc)).astype(np.float32)
    return [torch.from_numpy(x) for x in (g, a, b, c)]


def _check_bwd(op1, op2, g, a, b, c, got, what):
    ref = oracle.chain_bwd(op1, op2, g, a, b, c)
    n_out = g.numel()
    t_full = int(np.prod(np.broadcast_shapes(tuple(a.shape), tuple(b.shape)))) == n_out
    for k, (x, name) in enumerate(zip((a, b, c), "abc")):
        full = x.numel() == n_out
        exact = full and ((k == 0 and t_full) or (k == 1 and t_full and op1 != "div") or
                          (k == 2 and op2 != "div"))
        gv, rv = got[k].cpu().numpy(), ref[k]
        if exact:
            bitexact(gv, rv, f"{what} grad_{name}")
        else:
            within(gv, rv, ref[3 + k], f"{what} grad_{name}")


# ----------------------------------------------------------- forward

FWD_SHAPES = [((3, 97, 772), (772,), (772,)), ((2, 3, 131, 131), (1, 1, 131, 131), (1,)),
              ((5, 67, 203), (1, 67, 1), (5, 1, 203)), ((333,), (1,), (7, 333)),
              ((4, 1, 6), (5, 1), (1, 6)), ((2, 3, 4, 5, 2, 3, 2, 4), (4, 5, 1, 3, 2, 1), (1,))]


@pytest.mark.parametrize("op1", OPS)
def test_chain_forward_bit_exact(op1):
    rng = np.random.default_rng(800 + OPS.index(op1))
    for op2 in OPS:
        for sa, sb, sc in FWD_SHAPES:
            _, a, b, c = _inputs(rng, op1, op2, sa, sb, sc)
            got = zr.zr_chain_fwd(op1, op2, a.cuda(), b.cuda(), c.cuda()).cpu().numpy()
            bitexact(got, oracle.chain_fwd(op1, op2, a, b, c), f"chain fwd {op1} {op2} {sa} {sb} {sc}")


def test_chain_forward_strided_and_in_place():
    rng = np.random.default_rng(81)
    store = torch.from_numpy(rng.standard_normal((96, 40)).astype(np.float32))
    a = store.t()  # [40, 96], transposed view
    b = torch.from_numpy(rng.standard_normal((96,)).astype(np.float32))
    c = torch.from_numpy(rng.standard_normal((40, 1)).astype(np.float32))
    ref = oracle.chain_fwd("mul", "sub", a, b, c)
    got = zr.zr_chain_fwd("mul", "sub", to_gpu(a), b.cuda(), c.cuda()).cpu().numpy()
    bitexact(got, ref, "chain fwd transposed input")
    out_store = torch.empty((96, 40), device="cuda")
    zr.zr_chain_fwd("mul", "sub", to_gpu(a), b.cuda(), c.cuda(), out=out_store.t())
    bitexact(out_store.t().cpu().numpy(), ref, "chain fwd strided output")
    x = torch.from_numpy(rng.standard_normal((64, 96)).astype(np.float32))
    k = torch.from_numpy(_nonzero(rng, (1,)))
    ref = oracle.chain_fwd("add", "div", x, b, k)
    xd = x.cuda()
    # In place on a (same layout): each element is read before it is written.
    zr.zr_chain_fwd("add", "div", xd, b.cuda(), k.cuda(), out=xd)
    bitexact(xd.cpu().numpy(), ref, "chain fwd in place")


# ----------------------------------------------------------- backward

FUSED_SHAPES = [((3, 97, 772), (772,), (772,)),           # affine, c shaped like b
                ((2, 3, 131, 132), (1, 1, 131, 132), (1,)),  # scaled mask, c one element
                ((64, 1000), (1000,), (1000,)),
                ((5, 7, 300), (7, 300), (1, 1, 1))]
COMPOSED_SHAPES = [((16, 64, 96), (96,), (64, 1)),       # c shaped differently
                   ((96,), (32, 96), (32, 96)),          # a broadcast
                   ((5, 67, 203), (1, 67, 1), (5, 1, 203)),
                   ((4, 1, 6), (5, 1), (1, 6)),          # a broadcast on a middle dim
                   ((5, 6), (6,), (3, 5, 6)),            # t broadcast by c
                   ((7, 9), (7, 9), (1,))]                # b not reduced


@pytest.mark.parametrize("op1", OPS)
def test_chain_backward_fused_route(op1):
    rng = np.random.default_rng(900 + OPS.index(op1))
    for op2 in OPS:
        for sa, sb, sc in FUSED_SHAPES:
            g, a, b, c = _inputs(rng, op1, op2, sa, sb, sc)
            dev = [x.cuda() for x in (g, a, b, c)]
            grads = [torch.empty(s, device="cuda") for s in (sa, sb, sc)]
            assert _route(op1, op2, *dev, grads) == "fused", (op1, op2, sa, sb, sc)
            got = zr.zr_chain_bwd(op1, op2, *dev, grads=grads)
            _check_bwd(op1, op2, g, a, b, c, got, f"fused {op1} {op2} {sa} {sb} {sc}")
            again = zr.zr_chain_bwd(op1, op2, *dev)
            for u, v in zip(got, again):
                assert torch.equal(u.view(torch.int32), v.view(torch.int32))


@pytest.mark.parametrize("op1", OPS)
def test_chain_backward_composed_route(op1):
    rng = np.random.default_rng(950 + OPS.index(op1))
    for op2 in OPS:
        for sa, sb, sc in COMPOSED_SHAPES:
            g, a, b, c = _inputs(rng, op1, op2, sa, sb, sc)
            dev = [x.cuda() for x in (g, a, b, c)]
            grads = [torch.empty(s, device="cuda") for s in (sa, sb, sc)]
            assert _route(op1, op2, *dev, grads) == "composed", (op1, op2, sa, sb, sc)
            got = zr.zr_chain_bwd(op1, op2, *dev, grads=grads)
            _check_bwd(op1, op2, g, a, b, c, got, f"composed {op1} {op2} {sa} {sb} {sc}")


def test_chain_backward_partial_requests_and_empty():
    rng = np.random.default_rng(990)
    g, a, b, c = _inputs(rng, "mul", "div", (3, 97, 772), (772,), (772,))
    dev = [x.cuda() for x in (g, a, b, c)]
    ref = oracle.chain_bwd("mul", "div", g, a, b, c)
    for want in ((1, 0, 0), (0, 1, 0), (0, 0, 1), (1, 1, 0), (0, 1, 1)):
        got = zr.zr_chain_bwd("mul", "div", *dev, want=want)
        for k in range(3):
            if want[k]:
                what = f"partial {want} grad_{'abc'[k]}"
                if k == 0:
                    bitexact(got[k].cpu().numpy(), ref[k], what)
                else:
                    within(got[k].cpu().numpy(), ref[k], ref[3 + k], what)
            else:
                assert got[k] is None
    # Empty grad_out: reduced gradients are zero.
    ge = torch.empty((0, 5), device="cuda")
    ae = torch.empty((0, 5), device="cuda")
    got = zr.zr_chain_bwd("mul", "add", ge, ae, torch.ones(5, device="cuda"),
                          torch.ones(5, device="cuda"))
    assert got[0].numel() == 0 and torch.all(got[1] == 0) and torch.all(got[2] == 0)


@pytest.mark.parametrize("name,op1,op2,keys,dims,route", [
    ("c3", "mul", "add", ("g", "x", "gamma", "beta"), None, "fused"),
    # 131 columns rule out 16-byte vectors: the composed route; 132 allow them.
    ("c4", "add", "div", ("g", "scores", "mask", "scalar"), None, "composed"),
    ("c4", "add", "div", ("g", "scores", "mask", "scalar"), dict(N=2, H=3, T=132), "fused"),
])
def test_chain_workloads_small(name, op1, op2, keys, dims, route):
    host = workloads.make_inputs(name, **(dims or workloads.small_dims(name)))
    g, a, b, c = (host[k] for k in keys)
    dev = [x.cuda() for x in (g, a, b, c)]
    bitexact(zr.zr_chain_fwd(op1, op2, *dev[1:]).cpu().numpy(), oracle.chain_fwd(op1, op2, a, b, c),
             f"{name} chain fwd")
    grads = [torch.empty(x.shape, device="cuda") for x in (a, b, c)]
    assert _route(op1, op2, *dev, grads) == route
    got = zr.zr_chain_bwd(op1, op2, *dev, grads=grads)
    _check_bwd(op1, op2, g, a, b, c, got, f"{name} chain")


@pytest.mark.parametrize("name,op1,op2,keys", [
    ("c3", "mul", "add", ("g", "x", "gamma", "beta")),
    ("c4", "add", "div", ("g", "scores", "mask", "scalar")),
])
def test_chain_workloads_full_sampled(name, op1, op2, keys):
    """Full-size inputs in the launch configuration the benchmark uses;
    sampled outputs from the oracle, computed one by one."""
    rng = np.random.default_rng(11)
    host = workloads.make_inputs(name)
    g, a, b, c = (host[k] for k in keys)
    dev = [x.cuda() for x in (g, a, b, c)]
    out = zr.zr_chain_fwd(op1, op2, *dev[1:]).reshape(-1).cpu().numpy()
    n = out.size
    idx = np.unique(np.concatenate([rng.integers(0, n, 4000), [0, n - 1]])).astype(np.int64)
    t = oracle.binary_fwd(op1, a, b)
    bitexact(out[idx], oracle.binary_fwd_at(op2, t, c, idx), f"{name} chain fwd (sampled)")
    got = zr.zr_chain_bwd(op1, op2, *dev)
    for k, x in enumerate((a, b, c)):
        m = x.numel()
        idx = np.arange(m, dtype=np.int64) if m <= 4096 else np.unique(
            np.concatenate([rng.integers(0, m, 2000), [0, m - 1]])).astype(np.int64)
        vals, sabs = oracle.chain_bwd_at(op1, op2, k, g, a, b, c, idx)
        gv = got[k].reshape(-1).cpu().numpy()[idx]
        what = f"{name} chain grad_{'abc'[k]} (sampled)"
        if k == 0:
            bitexact(gv, vals, what)
        else:
            within(gv, vals, sabs, what)


def _dev_view(x, strides):
    """Device view of x's values with the given element strides (inside a
    larger zero-filled buffer)."""
    span = 1 + sum((n - 1) * s for n, s in zip(x.shape, strides))
    buf = torch.zeros(span, device="cuda")
    v = buf.as_strided(x.shape, strides)
    v.copy_(x.cuda())
    return v


STRIDED = [
    # grad_out and a stepped along the inner dim: fused route.
    ("fused", (6, 40, 132), (132,), (132,), {"g": (40 * 264, 264, 2), "a": (40 * 264, 264, 2)}),
    # a with permuted outer dims: fused route.
    ("fused", (6, 40, 132), (132,), (132,), {"a": (132, 6 * 132, 1)}),
    # scaled-mask layout with a stepped a: fused route, one-element c.
    ("fused", (2, 3, 131, 132), (1, 1, 131, 132), (1,), {"a": (3 * 131 * 264, 131 * 264, 264, 2)}),
    # b and c stepped: c is not in b's dense layout, composed route.
    ("composed", (6, 40, 132), (132,), (132,), {"b": (2,), "c": (2,)}),
]


@pytest.mark.parametrize("route,sa,sb,sc,st", STRIDED)
def test_chain_backward_strided_views(route, sa, sb, sc, st):
    """Strided and stepped views of grad_out, a, b and c, on both routes:
    the same results as dense copies of the same values."""
    rng = np.random.default_rng(996)
    for op1 in OPS:
        for op2 in OPS:
            g, a, b, c = _inputs(rng, op1, op2, sa, sb, sc)
            dev = []
            for name, x in zip("gabc", (g, a, b, c)):
                dev.append(_dev_view(x, st[name]) if name in st else x.cuda())
            grads = [torch.empty(s, device="cuda") for s in (sa, sb, sc)]
            assert _route(op1, op2, *dev, grads) == route, (op1, op2, sa, st)
            got = zr.zr_chain_bwd(op1, op2, *dev, grads=grads)
            _check_bwd(op1, op2, g, a, b, c, got, f"strided {route} {op1} {op2} {sa} {st}")
