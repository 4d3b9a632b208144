"""GPU parity of the bfloat16-storage entry points (zr_binary_fwd_t,
zr_binary_bwd_t, zr_sum_to_shape_t with ZR_BF16) against the CPU oracle.

The oracle reads the same bf16 values (as binary32), computes as for float
storage and rounds every stored result once to bf16.  Forward outputs and
one-operation gradients must be bit-identical; summed gradients within
1e-5 * sum|terms| + 2^-7 * |value| per element: a sum within the float
tolerance can still round to the bf16 neighbour of the exact sum's rounding
when the two fall on either side of a rounding boundary, one bf16 unit in
the last place (at most 2^-7 of the value).  Chained steps read the bf16
intermediate, as the GPU does.
"""
import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads
from parity import bitexact, within

pytestmark = pytest.mark.gpu

OPS = ["add", "sub", "mul", "div"]
BINARY = ["c1", "c2", "c3", "c4", "c5a", "c5b", "x1"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


def _bf(x):
    """bf16-rounded copy of a float32 CPU tensor, keeping its strides."""
    st = x.untyped_storage()
    flat = torch.empty(0, dtype=x.dtype).set_(st, 0, (st.nbytes() // 4,), (1,))
    r = torch.from_numpy(oracle.round_bf16(flat.numpy()))
    return r.as_strided(x.shape, x.stride(), x.storage_offset())


def _dev16(x):
    """Device bf16 tensor with x's values (x already bf16-representable) and strides."""
    st = x.untyped_storage()
    flat = torch.empty(0, dtype=x.dtype).set_(st, 0, (st.nbytes() // 4,), (1,))
    d = flat.to(torch.bfloat16).cuda()
    return d.as_strided(x.shape, x.stride(), x.storage_offset())


def _f32(t):
    return t.float().cpu().numpy()


def _check_grad(got, ref, sabs, exact, what):
    if exact:
        bitexact(got, ref, what)
    else:
        r64 = np.asarray(ref, np.float64)
        within(got, ref, sabs + 2.0 ** -7 / 1e-5 * np.abs(r64), what)


@pytest.mark.parametrize("name", BINARY)
def test_bf16_workloads_small(name):
    host = {k: _bf(v) for k, v in workloads.make_inputs(name, **workloads.small_dims(name)).items()}
    gpu = {k: _dev16(v) for k, v in host.items()}
    ref = dict(host)
    for step in workloads.STEPS[name]:
        if step[0] == "fwd":
            _, op, an, bn, on = step
            gpu[on] = zr.zr_binary_fwd(op, gpu[an], gpu[bn])
            assert gpu[on].dtype == torch.bfloat16
            ref[on] = torch.from_numpy(oracle.round_bf16(oracle.binary_fwd(op, ref[an], ref[bn])))
            bitexact(_f32(gpu[on]), ref[on].numpy(), f"bf16 {name} fwd {op}")
        else:
            _, op, gn, an, bn, gan, gbn = step
            ga, gb = zr.zr_binary_bwd(op, gpu[gn], gpu[an], gpu[bn])
            ra, rb, sa, sb = oracle.binary_bwd(op, ref[gn], ref[an], ref[bn])
            n_out = ref[gn].numel()
            for w, got, r, sab in ((0, ga, ra, sa), (1, gb, rb, sb)):
                reduced = r.size != n_out
                exact = not reduced and not (op == "div" and w == 1)
                _check_grad(_f32(got), oracle.round_bf16(r), sab, exact,
                            f"bf16 {name} bwd {op} grad_{'ab'[w]}")
            gpu[gan], gpu[gbn] = ga, gb
            ref[gan] = torch.from_numpy(oracle.round_bf16(ra))
            ref[gbn] = torch.from_numpy(oracle.round_bf16(rb))


@pytest.mark.parametrize("op", OPS)
def test_bf16_random_views(op):
    rng = np.random.default_rng(1500 + OPS.index(op))
    for it in range(40):
        nd = int(rng.integers(1, 5))
        out = tuple(int(v) for v in rng.integers(1, 9, nd))
        sa = tuple(s if rng.random() < 0.7 else 1 for s in out)
        sb = tuple(s if rng.random() < 0.5 else 1 for s in out)[int(rng.integers(0, nd)):]
        # a: sometimes a transposed or offset view
        base = torch.from_numpy(rng.standard_normal(int(np.prod(sa)) + 3).astype(np.float32))
        off = int(rng.integers(0, 4))
        a = base[off:off + int(np.prod(sa))].reshape(sa)
        if nd >= 2 and rng.random() < 0.5:
            a = torch.from_numpy(rng.standard_normal(sa[::-1]).astype(np.float32)).permute(
                *reversed(range(nd)))
        b = torch.from_numpy(rng.standard_normal(sb).astype(np.float32))
        if op == "div":
            b = torch.sign(b) * (0.5 + b.abs())
        a, b = _bf(a), _bf(b)
        g = _bf(torch.from_numpy(rng.standard_normal(np.broadcast_shapes(sa, sb)).astype(np.float32)))
        out_gpu = zr.zr_binary_fwd(op, _dev16(a), _dev16(b))
        bitexact(_f32(out_gpu), oracle.round_bf16(oracle.binary_fwd(op, a, b)), f"bf16 fwd {op} {sa} {sb}")
        ga, gb = zr.zr_binary_bwd(op, _dev16(g), _dev16(a), _dev16(b))
        ra, rb, s1, s2 = oracle.binary_bwd(op, g, a, b)
        n_out = g.numel()
        for w, got, r, sab in ((0, ga, ra, s1), (1, gb, rb, s2)):
            exact = r.size == n_out and not (op == "div" and w == 1)
            _check_grad(_f32(got), oracle.round_bf16(r), sab, exact, f"bf16 bwd {op} {sa} {sb} {w}")


def test_bf16_sum_to_shape_and_mixed_types():
    rng = np.random.default_rng(1600)
    for shape, tgt in (((4096, 1024), (1024,)), ((64, 300, 256), (1, 300, 1)), ((33, 65), (33, 65)),
                       (((1 << 20) + 3,), (1,)), ((700, 20000), (20000,))):
        x = _bf(torch.from_numpy(rng.standard_normal(shape).astype(np.float32)))
        got = zr.zr_sum_to_shape(_dev16(x), tgt)
        assert got.dtype == torch.bfloat16
        ref, sabs = oracle.sum_to_shape(x, tgt)
        _check_grad(_f32(got), oracle.round_bf16(ref), sabs, int(np.prod(tgt)) == x.numel(),
                    f"bf16 sum {shape}->{tgt}")
    with pytest.raises(TypeError):
        zr.zr_binary_fwd("add", torch.ones(4, device="cuda"), torch.ones(4, device="cuda", dtype=torch.bfloat16))


WIDE = [((333, 1024), (1024,)), ((7, 40, 96), (1, 40, 1)), ((24, 1, 64), (1, 16, 64)),
        ((2, 3, 136, 136), (1, 1, 136, 136)), ((64, 1000), (64, 1000))]


@pytest.mark.parametrize("op", OPS)
def test_bf16_wide_vectors(op):
    """Shapes whose rows allow 16-byte bf16 vectors (8 elements), against
    the oracle: forward bit-exact, gradients as above."""
    rng = np.random.default_rng(1700 + OPS.index(op))
    for sa, sb in WIDE:
        a = _bf(torch.from_numpy(rng.standard_normal(sa).astype(np.float32)))
        b = torch.from_numpy(rng.standard_normal(sb).astype(np.float32))
        if op == "div":
            b = torch.sign(b) * (0.5 + b.abs())
        b = _bf(b)
        g = _bf(torch.from_numpy(rng.standard_normal(np.broadcast_shapes(sa, sb)).astype(np.float32)))
        out = zr.zr_binary_fwd(op, _dev16(a), _dev16(b))
        bitexact(_f32(out), oracle.round_bf16(oracle.binary_fwd(op, a, b)), f"bf16 wide fwd {op} {sa} {sb}")
        ga, gb = zr.zr_binary_bwd(op, _dev16(g), _dev16(a), _dev16(b))
        ra, rb, s1, s2 = oracle.binary_bwd(op, g, a, b)
        for w, got, r, sab in ((0, ga, ra, s1), (1, gb, rb, s2)):
            exact = r.size == g.numel() and not (op == "div" and w == 1)
            _check_grad(_f32(got), oracle.round_bf16(r), sab, exact, f"bf16 wide bwd {op} {sa} {sb} {w}")


def test_bf16_division_equals_ieee_divide_on_every_pair():
    """The divisions bf16 storage uses, over all 2^32 ordered pairs of
    bfloat16 bit patterns (normals, subnormals, zeros, infinities, NaNs):
    the exact one (approximate quotient plus one correction with the exact
    residual) gives the IEEE binary32 quotient bit for bit; the one for
    stored results (product with the approximate reciprocal) rounds to the
    same bfloat16 number as the IEEE quotient."""
    import ctypes
    L = zr.lib()
    L.zr_test_div_short_check.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    out = torch.tensor([0, -1, 0, -1], dtype=torch.int64, device="cuda")
    rc = L.zr_test_div_short_check(out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    res = out.tolist()
    for k, what in enumerate(("exact binary32 quotient", "quotient rounded to bf16")):
        bad, first = res[2 * k], res[2 * k + 1] & ((1 << 64) - 1)
        assert bad == 0, (f"{what}: {bad} pairs differ; first x bits 0x{first >> 16:04x}, "
                          f"y bits 0x{first & 0xffff:04x}")


def test_bf16_division_of_the_scores_workload_full_size():
    """c4's scores [8,12,1024,1024] in bf16 divided by [8.0] at full size (the
    plan the benchmark times): bit-identical to the oracle on sampled
    elements."""
    host = workloads.make_inputs("c4h")
    t = _bf(host["scores"])
    d_t, d_s = _dev16(t), _dev16(_bf(host["scalar"]))
    out = zr.zr_binary_fwd("div", d_t, d_s)
    rng = np.random.default_rng(1500)
    idx = np.sort(rng.choice(t.numel(), 4096, replace=False)).astype(np.int64)
    want = oracle.round_bf16(oracle.binary_fwd_at("div", t, _bf(host["scalar"]), idx))
    bitexact(_f32(out).reshape(-1)[idx], want, "c4h t / 8")


# GeLU in bf16 evaluates erfc with a shorter fitted polynomial (relative error
# below 2^-16.3): the summed terms may carry 2^-14 of their size (in units of
# the binary32 bound's 2^-24: 2^10).
_SHORT = 2.0 ** 10


def _ulp_bf16(v):
    """One bf16 unit in the last place of |v| (normal range; subnormal spacing
    below 2^-126)."""
    v = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(v)
    return np.where(v >= 2.0 ** -126, np.ldexp(1.0, e - 8), 2.0 ** -133)


def test_bf16_gelu_on_every_bf16_input():
    """GeLU forward and backward (grad_out = 1) on all 65536 bf16 bit
    patterns: each result is within half a bf16 unit of the exact value plus
    2^-14 of the terms' size (the shorter erfc and binary32 rounding) plus
    2^-120, so it is the correctly rounded value except next to a rounding
    boundary; NaN where the exact result is NaN, infinities equal."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = torch.from_numpy(bits.view(np.float32).copy())
    xd = x.to(torch.bfloat16).cuda()
    ones = torch.ones(65536, dtype=torch.bfloat16, device="cuda")
    for what, got, ref, mag in (
            ("fwd", _f32(zr.zr_unary_fwd("gelu", xd)), oracle.unary_fwd("gelu", x), None),
            ("bwd", _f32(zr.zr_unary_bwd("gelu", ones, xd)), *oracle.unary_bwd("gelu", torch.ones(65536), x))):
        got = got.astype(np.float64)
        ref = ref.astype(np.float64)
        gn, rn = np.isnan(got), np.isnan(ref)
        assert np.array_equal(gn, rn), f"gelu {what}: NaN positions differ"
        fin = ~gn & np.isfinite(ref)
        assert np.array_equal(got[~gn & ~fin], ref[~gn & ~fin]), f"gelu {what}: infinities differ"
        size = np.abs(ref) if mag is None else np.asarray(mag, np.float64)
        allowed = 0.5 * _ulp_bf16(ref[fin]) + 2.0 ** -14 * size[fin] + 2.0 ** -120
        err = np.abs(got[fin] - ref[fin])
        bad = np.nonzero(err > allowed)[0]
        assert bad.size == 0, (f"gelu {what}: {bad.size} inputs beyond the bound; first x = "
                               f"{x.numpy()[fin][bad[0]]!r}: gpu {got[fin][bad[0]]!r} "
                               f"exact {ref[fin][bad[0]]!r}")
        # Away from rounding boundaries the result is the correctly rounded one.
        exact16 = oracle.round_bf16(ref.astype(np.float32)).astype(np.float64)
        assert np.mean(got[fin] == exact16[fin]) > 0.98, f"gelu {what}: too many off by one unit"


def test_unary_ops_in_bf16():
    """scale and GeLU on bf16 storage (zr_unary_fwd_t / zr_unary_bwd_t):
    scale is bit-identical to the exact product rounded to bf16; GeLU is
    within the binary32 bound plus one bf16 unit (2^-7 of the value).
    Shapes with 8-wide rows, ragged rows, a strided view, tails and special
    values."""
    from parity import gelu_close
    rng = np.random.default_rng(1600)
    xs = [rng.standard_normal((96, 1024)) * 3, rng.standard_normal((64, 1031)) * 3,
          np.linspace(-14, 14, 8000),
          np.array([0.0, -0.0, 1e-40, -1e-40, -0.7518, 88.0, -88.0, np.inf, -np.inf, np.nan])]
    for x in xs:
        xt = _bf(torch.from_numpy(x.astype(np.float32)))
        g = _bf(torch.from_numpy(rng.standard_normal(x.shape).astype(np.float32)))
        xd, gd = _dev16(xt), _dev16(g)
        for alpha in (0.125, -3.0):
            got = _f32(zr.zr_unary_fwd("scale", xd, alpha=alpha))
            bitexact(got, oracle.round_bf16(oracle.unary_fwd("scale", xt, alpha=alpha)),
                     f"bf16 scale fwd {x.shape} {alpha}")
            got = _f32(zr.zr_unary_bwd("scale", gd, None, alpha=alpha))
            bitexact(got, oracle.round_bf16(oracle.unary_bwd("scale", g, None, alpha=alpha)[0]),
                     f"bf16 scale bwd {x.shape} {alpha}")
        xv = xt.numpy().astype(np.float64)
        widen = 2.0 ** 17 / (16.0 + 2.0 * xv ** 2)  # 2^-7 |value| in units of the bound
        ref = oracle.unary_fwd("gelu", xt)
        got = _f32(zr.zr_unary_fwd("gelu", xd))
        with np.errstate(all="ignore"):
            mag = np.abs(ref.astype(np.float64))
            gelu_close(got, ref, xv, mag * (1.0 + widen), f"bf16 gelu fwd {x.shape}")
        gref, gmag = oracle.unary_bwd("gelu", g, xt)
        got = _f32(zr.zr_unary_bwd("gelu", gd, xd))
        with np.errstate(all="ignore"):
            gelu_close(got, gref, xv, gmag * (1.0 + _SHORT / (16.0 + 2.0 * xv ** 2))
                       + np.abs(gref.astype(np.float64)) * widen, f"bf16 gelu bwd {x.shape}")
    # A strided bf16 view, written into a strided bf16 output.
    base = _bf(torch.from_numpy((rng.standard_normal((96, 33, 2)) * 2).astype(np.float32)))
    xv_t = base[:, :, 1].t()
    out_store = torch.zeros((96, 33), dtype=torch.bfloat16, device="cuda")
    zr.zr_unary_fwd("scale", _dev16(xv_t), alpha=0.5, out=out_store.t())
    bitexact(_f32(out_store.t()), oracle.round_bf16(oracle.unary_fwd("scale", xv_t, alpha=0.5)),
             "bf16 scale strided")


def test_unary_workload_in_bf16_full_size():
    """u1 in bf16 at full size ([16384, 3072], 8-wide plans): GeLU and scale
    forward and backward on sampled elements (the ops are elementwise, so the
    oracle evaluates the sampled inputs alone)."""
    from parity import gelu_close
    host = workloads.make_inputs("u1h")
    x, g = _bf(host["x"]), _bf(host["g"])
    xd, gd = _dev16(x), _dev16(g)
    rng = np.random.default_rng(1601)
    idx = np.unique(rng.integers(0, x.numel(), 8192))
    xs = torch.from_numpy(x.reshape(-1).numpy()[idx])
    gs = torch.from_numpy(g.reshape(-1).numpy()[idx])
    xv = xs.numpy().astype(np.float64)
    widen = 2.0 ** 17 / (16.0 + 2.0 * xv ** 2)
    h = _f32(zr.zr_unary_fwd("gelu", xd)).reshape(-1)[idx]
    ref = oracle.unary_fwd("gelu", xs)
    gelu_close(h, ref, xv, np.abs(ref.astype(np.float64)) * (1.0 + widen), "u1h gelu fwd")
    gx = _f32(zr.zr_unary_bwd("gelu", gd, xd)).reshape(-1)[idx]
    gref, gmag = oracle.unary_bwd("gelu", gs, xs)
    gelu_close(gx, gref, xv, gmag * (1.0 + _SHORT / (16.0 + 2.0 * xv ** 2))
               + np.abs(gref.astype(np.float64)) * widen, "u1h gelu bwd")
    s = _f32(zr.zr_unary_fwd("scale", xd, alpha=0.125)).reshape(-1)[idx]
    bitexact(s, oracle.round_bf16(oracle.unary_fwd("scale", xs, alpha=0.125)), "u1h scale fwd")
