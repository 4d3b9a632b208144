"""GPU tests of GeLU on bfloat16 storage read from a table (k_gelu_bf16).

Large flat bfloat16 GeLU calls take their results from a table in shared
memory that each CTA fills with the arithmetic path's own functors, and
evaluate the elements outside it (|x| < 2^-24, |x| >= 256, infinities, NaN)
in place.  So they must equal the arithmetic path bit for bit, on every
bfloat16 input and every layout the flat plans take.  The arithmetic path is
run on the same values in pieces below the table's size limit; it is pinned
to the oracle on every bfloat16 input in test_gpu_bf16.py, and the first
copy of those inputs is checked against the oracle's bound here as well.
"""
import ctypes
import json

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle

pytestmark = pytest.mark.gpu

LIMIT = 152 * 32768  # elements from which flat bfloat16 GeLU reads the table


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    lib = zr.lib()
    lib.zr_test_describe_unary_t.argtypes = [ctypes.c_int, ctypes.c_int, zr.ZrTensor,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_char_p, ctypes.c_size_t]
    return lib


def _kernel(L, x, out, g=None):
    """The kernel the unary entry point launches for these tensors."""
    buf = ctypes.create_string_buffer(4096)
    dx, kx = zr._desc(x)
    ost = zr._i64(out.stride())
    if g is None:
        rc = L.zr_test_describe_unary_t(1, 1, dx, None, out.data_ptr(),
                                        ctypes.cast(ost, ctypes.c_void_p), buf, len(buf))
    else:
        dg, kg = zr._desc(g)
        rc = L.zr_test_describe_unary_t(1, 1, dg, ctypes.addressof(dx), out.data_ptr(),
                                        ctypes.cast(ost, ctypes.c_void_p), buf, len(buf))
    assert rc == 0, rc
    return json.loads(buf.value.decode())["kernel"]


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _arith(L, xs, gs=None):
    """GeLU (gs None) or its backward through the arithmetic path: flat pieces
    of fewer than LIMIT elements of contiguous copies."""
    xs = xs.contiguous().reshape(-1)
    gs = None if gs is None else gs.contiguous().reshape(-1)
    out = torch.empty_like(xs)
    step = LIMIT // 2
    for s in range(0, xs.numel(), step):
        xp = xs[s:s + step]
        op = out[s:s + step]
        if gs is None:
            assert _kernel(L, xp, op) == "flat"
            zr.zr_unary_fwd("gelu", xp, out=op)
        else:
            assert _kernel(L, xp, op, gs[s:s + step]) == "flat"
            zr.zr_unary_bwd("gelu", gs[s:s + step], xp, grad_x=op)
    return out


def _every_pattern(copies):
    """All 65536 bfloat16 patterns, `copies` times, as a [copies, 65536]
    device tensor, each copy in another order."""
    rng = np.random.default_rng(1700)
    bits = np.stack([rng.permutation(65536) for _ in range(copies)]).astype(np.uint16)
    bits[0] = np.arange(65536, dtype=np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _ulp_bf16(v):
    v = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(v)
    return np.where(v >= 2.0 ** -126, np.ldexp(1.0, e - 8), 2.0 ** -133)


def test_table_equals_arithmetic_on_every_bf16_input(L):
    """Forward and backward over 160 permuted copies of every bfloat16 pattern
    (10.5 M elements): bit for bit the arithmetic path's results."""
    x = _every_pattern(160)
    torch.manual_seed(1701)
    g = (torch.randn(x.shape, device="cuda") * 2).to(torch.bfloat16)
    y = torch.empty_like(x)
    assert _kernel(L, x, y) == "gelu_table"
    zr.zr_unary_fwd("gelu", x, out=y)
    ref = _arith(L, x)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y).reshape(-1), _bits(ref)), "table forward differs"
    gx = torch.empty_like(x)
    assert _kernel(L, x, gx, g) == "gelu_table"
    zr.zr_unary_bwd("gelu", g, x, grad_x=gx)
    ref = _arith(L, x, g)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(gx).reshape(-1), _bits(ref)), "table backward differs"
    # The first copy (every pattern in order) against the oracle's bound.
    xh = x[0].float().cpu()
    got = y[0].float().cpu().numpy().astype(np.float64)
    exact = oracle.unary_fwd("gelu", xh).astype(np.float64)
    fin = np.isfinite(exact) & ~np.isnan(got)
    assert np.array_equal(np.isnan(got), np.isnan(exact))
    allowed = 0.5 * _ulp_bf16(exact[fin]) + 2.0 ** -14 * np.abs(exact[fin]) + 2.0 ** -120
    assert np.all(np.abs(got[fin] - exact[fin]) <= allowed)


@pytest.mark.parametrize("layout", ["odd", "four", "row_strided", "col_strided", "expanded",
                                    "in_place"])
def test_table_layouts(L, layout):
    """The flat layouts: 1-element items (odd size), 4-element items, rows
    with a stride (staged 16-byte vectors), a column-strided view (2-byte
    gathers), a column broadcast along rows (8-wide vectors of one loaded
    element: not staged), and in place; normally distributed inputs with a
    few out-of-table values planted."""
    torch.manual_seed(1702)
    n = LIMIT + 12345
    if layout == "odd":
        base = torch.randn(n | 1, device="cuda")
        x = base.to(torch.bfloat16)
    elif layout == "four":
        x = torch.randn(n - n % 8 + 4, device="cuda").to(torch.bfloat16)
    elif layout == "row_strided":
        x = torch.randn(1300, 8200, device="cuda").to(torch.bfloat16)[:, :8192]
    elif layout == "col_strided":
        x = torch.randn(1300, 16384, device="cuda").to(torch.bfloat16)[:, ::2]
    elif layout == "expanded":
        x = torch.randn(1300, 1, device="cuda").to(torch.bfloat16).expand(1300, 8192)
    else:
        x = torch.randn(1300, 8192, device="cuda").to(torch.bfloat16)
    flat = x.reshape(-1) if x.is_contiguous() else None
    special = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 300.0, -300.0, float("inf"),
                            float("-inf"), float("nan"), 2.0 ** -24, -(2.0 ** -24), 255.9],
                           dtype=torch.bfloat16, device="cuda")
    if flat is not None:
        flat[1000:1000 + special.numel()] = special
    elif layout == "expanded":
        x = x.contiguous()[:, :1].clone()
        x[100:100 + special.numel(), 0] = special
        x = x.expand(1300, 8192)
    else:
        x[7, 100:100 + special.numel()] = special
    g = torch.randn(x.shape, device="cuda").to(torch.bfloat16)
    xs, gs = x.clone(), g.clone()  # contiguous copies for the arithmetic path
    ref_f = _arith(L, xs)
    ref_b = _arith(L, xs, gs)
    if layout == "in_place":
        assert _kernel(L, x, x) == "gelu_table"
        zr.zr_unary_fwd("gelu", x, out=x)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(x).reshape(-1), _bits(ref_f)), "in place forward"
        x.copy_(xs)
        assert _kernel(L, x, x, g) == "gelu_table"
        zr.zr_unary_bwd("gelu", g, x, grad_x=x)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(x).reshape(-1), _bits(ref_b)), "in place backward"
        return
    y = torch.empty(x.shape, dtype=torch.bfloat16, device="cuda")
    assert _kernel(L, x, y) == "gelu_table"
    zr.zr_unary_fwd("gelu", x, out=y)
    gx = torch.empty(x.shape, dtype=torch.bfloat16, device="cuda")
    assert _kernel(L, x, gx, g) == "gelu_table"
    zr.zr_unary_bwd("gelu", g, x, grad_x=gx)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y).reshape(-1), _bits(ref_f)), f"{layout} forward"
    assert np.array_equal(_bits(gx).reshape(-1), _bits(ref_b)), f"{layout} backward"


def test_table_output_strided(L):
    """A contiguous input written into rows with a stride (the output's
    layout decides the flat plan's rows)."""
    torch.manual_seed(1703)
    x = torch.randn(1300, 8192, device="cuda").to(torch.bfloat16)
    store = torch.full((1300, 8200), 7.0, dtype=torch.bfloat16, device="cuda")
    y = store[:, :8192]
    assert _kernel(L, x, y) == "gelu_table"
    zr.zr_unary_fwd("gelu", x, out=y)
    ref = _arith(L, x)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y).reshape(-1), _bits(ref))
    assert torch.all(store[:, 8192:] == 7.0)  # the gaps between rows are untouched
