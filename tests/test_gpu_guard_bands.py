"""Out-of-bounds writes: every output and the workspace sit between guard
bands of a sentinel value, at misaligned element offsets, for odd sizes
(1, 3, 7, 33 per dim) and both element types; after each call the bands must
be intact and the results must match the oracle (forwards bit-exact,
summed gradients within tolerance)."""
import ctypes

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
from parity import bitexact, within

pytestmark = pytest.mark.gpu

SENTINEL = -7.25  # exact in binary32 and bf16
PAD = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


class Guarded:
    """A dense tensor of `shape` at element offset `off` inside a buffer
    whose other elements hold SENTINEL."""

    def __init__(self, shape, dtype, off):
        n = int(np.prod(shape)) if shape else 1
        self.buf = torch.full((PAD + off + n + PAD,), SENTINEL, dtype=dtype, device="cuda")
        self.lo, self.hi = PAD + off, PAD + off + n
        self.t = self.buf[self.lo:self.hi].view(shape)

    def intact(self):
        return bool(torch.all(self.buf[:self.lo] == SENTINEL)) and \
            bool(torch.all(self.buf[self.hi:] == SENTINEL))


def _round(x, dtype):
    return oracle.round_bf16(x) if dtype == torch.bfloat16 else x


def _shapes(rng):
    nd = int(rng.integers(1, 5))
    out = [int(v) for v in rng.choice([1, 3, 7, 33], nd)]
    sa = tuple(s if rng.random() < 0.7 else 1 for s in out)
    sb = tuple(s if rng.random() < 0.5 else 1 for s in out)[int(rng.integers(0, nd)):]
    return sa, sb


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_outputs_and_workspace_stay_in_bounds(dtype):
    rng = np.random.default_rng(1700 + (dtype == torch.bfloat16))
    ops = ["add", "sub", "mul", "div"]
    for it in range(60):
        sa, sb = _shapes(rng)
        op = ops[it % 4]
        out_shape = tuple(np.broadcast_shapes(sa, sb))
        a = rng.standard_normal(sa).astype(np.float32)
        b = (np.sign(rng.standard_normal(sb)) * (0.5 + rng.random(sb))).astype(np.float32)
        g = rng.standard_normal(out_shape).astype(np.float32)
        if dtype == torch.bfloat16:
            a, b, g = oracle.round_bf16(a), oracle.round_bf16(b), oracle.round_bf16(g)
        ad = torch.from_numpy(a).to(dtype).cuda()
        bd = torch.from_numpy(b).to(dtype).cuda()
        gd = torch.from_numpy(g).to(dtype).cuda()
        at, bt, gt = (torch.from_numpy(x) for x in (a, b, g))
        what = f"{dtype} {op} {sa} {sb}"
        # forward
        out = Guarded(out_shape, dtype, int(rng.integers(0, 9)))
        zr.zr_binary_fwd(op, ad, bd, out=out.t)
        torch.cuda.synchronize()
        assert out.intact(), f"fwd {what}: wrote outside its output"
        bitexact(out.t.float().cpu().numpy(), _round(oracle.binary_fwd(op, at, bt), dtype),
                 f"fwd {what}")
        # backward, both gradients, workspace guarded too
        ga = Guarded(sa, dtype, int(rng.integers(0, 9)))
        gb = Guarded(sb, dtype, int(rng.integers(0, 9)))
        dg, k1 = zr._desc(gd)
        da, k2 = zr._desc(ad)
        db, k3 = zr._desc(bd)
        need = ctypes.c_size_t(0)
        dt = zr.ZR_BF16 if dtype == torch.bfloat16 else zr.ZR_F32
        assert zr.lib().zr_binary_bwd_t(dt, zr.OPS[op], dg, da, db, ga.t.data_ptr(), gb.t.data_ptr(),
                                        None, ctypes.byref(need), None) == 0
        nws = max(16, need.value)
        wsbuf = torch.full((PAD + nws + PAD,), 0x5A, dtype=torch.uint8, device="cuda")
        ws = wsbuf[PAD:PAD + nws]  # 16-byte aligned: PAD is a multiple of 16
        zr.zr_binary_bwd(op, gd, ad, bd, grad_a=ga.t, grad_b=gb.t, workspace=ws)
        torch.cuda.synchronize()
        assert ga.intact() and gb.intact(), f"bwd {what}: wrote outside a gradient"
        assert bool(torch.all(wsbuf[:PAD] == 0x5A)) and bool(torch.all(wsbuf[PAD + nws:] == 0x5A)), \
            f"bwd {what}: wrote outside the workspace ({nws} bytes)"
        ra, rb, s1, s2 = oracle.binary_bwd(op, gt, at, bt)
        n_out = int(np.prod(out_shape))
        for w, (got, ref, sabs) in enumerate(((ga.t, ra, s1), (gb.t, rb, s2))):
            got = got.float().cpu().numpy()
            single = ref.size == n_out and not (op == "div" and w == 1)
            if single:
                bitexact(got, _round(ref, dtype), f"bwd {what} grad_{'ab'[w]}")
            else:
                slack = 2.0 ** -7 * np.abs(ref.astype(np.float64)) if dtype == torch.bfloat16 else 0.0
                within(got, ref, sabs + slack / 1e-5, f"bwd {what} grad_{'ab'[w]}")
        # sum-to-shape onto b's shape
        so = Guarded(sb, dtype, int(rng.integers(0, 9)))
        zr.zr_sum_to_shape(gd, sb, out=so.t)
        torch.cuda.synchronize()
        assert so.intact(), f"sum {what}: wrote outside its output"
        ref, sabs = oracle.sum_to_shape(gt, sb)
        slack = 2.0 ** -7 * np.abs(ref.astype(np.float64)) if dtype == torch.bfloat16 else 0.0
        within(so.t.float().cpu().numpy(), ref, sabs + slack / 1e-5, f"sum {what}")


def test_chain_and_unary_outputs_stay_in_bounds():
    rng = np.random.default_rng(1702)
    for it in range(24):
        n = int(rng.choice([1, 3, 7, 33]))
        m = int(rng.choice([1, 3, 7, 33, 132]))
        sa, sb, sc = (n, 5, m), (m,), ((m,) if it % 2 else (1,))
        a = torch.from_numpy(rng.standard_normal(sa).astype(np.float32))
        b = torch.from_numpy((0.5 + rng.random(sb)).astype(np.float32))
        c = torch.from_numpy((0.5 + rng.random(sc)).astype(np.float32))
        g = torch.from_numpy(rng.standard_normal(sa).astype(np.float32))
        op1, op2 = ["mul", "add", "div", "sub"][it % 4], ["add", "div", "mul", "sub"][(it // 4) % 4]
        out = Guarded(sa, torch.float32, int(rng.integers(0, 9)))
        zr.zr_chain_fwd(op1, op2, a.cuda(), b.cuda(), c.cuda(), out=out.t)
        grads = [Guarded(s, torch.float32, int(rng.integers(0, 9))) for s in (sa, sb, sc)]
        zr.zr_chain_bwd(op1, op2, g.cuda(), a.cuda(), b.cuda(), c.cuda(), grads=[x.t for x in grads])
        torch.cuda.synchronize()
        what = f"chain {op1} {op2} {sa} {sb} {sc}"
        assert out.intact() and all(x.intact() for x in grads), f"{what}: wrote out of bounds"
        bitexact(out.t.cpu().numpy(), oracle.chain_fwd(op1, op2, a, b, c), what)
        for dtype in (torch.float32, torch.bfloat16):
            x = a if dtype == torch.float32 else torch.from_numpy(oracle.round_bf16(a.numpy()))
            xd = x.to(dtype).cuda()
            for op in ("scale", "gelu"):
                u = Guarded(sa, dtype, int(rng.integers(0, 9)))
                zr.zr_unary_fwd(op, xd, alpha=0.5, out=u.t)
                ub = Guarded(sa, dtype, int(rng.integers(0, 9)))
                zr.zr_unary_bwd(op, g.to(dtype).cuda(), xd, alpha=0.5, grad_x=ub.t)
                torch.cuda.synchronize()
                assert u.intact() and ub.intact(), f"{op} {dtype} {sa}: wrote out of bounds"
