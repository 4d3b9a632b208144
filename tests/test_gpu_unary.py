"""GPU parity of the unary elementwise ops (zr_unary_fwd / zr_unary_bwd)
against the CPU oracle, through the C ABI.

scale: bit-identical (one binary32 multiply).  GeLU: within
(16 + 2x^2) * 2^-24 * |exact| + 2^-120 forward and
(16 + 2x^2) * 2^-24 * |g| (Phi(x) + |x| phi(x)) + 2^-120 backward, per
element (the oracle evaluates the exact definition in binary64).
"""
import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads
from parity import bitexact, gelu_close as _gelu_close, to_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


def test_scale_bit_exact_strided_and_in_place():
    rng = np.random.default_rng(40)
    base = torch.from_numpy(rng.standard_normal((300, 257)).astype(np.float32))
    x = base.t()
    for alpha in (0.125, -3.0, 1e-30):
        out = zr.zr_unary_fwd("scale", to_gpu(x), alpha=alpha).cpu().numpy()
        bitexact(out, oracle.unary_fwd("scale", x, alpha=alpha), f"scale fwd {alpha}")
        g = torch.from_numpy(rng.standard_normal((257, 300)).astype(np.float32))
        gx = zr.zr_unary_bwd("scale", g.cuda(), None, alpha=alpha).cpu().numpy()
        bitexact(gx, oracle.unary_bwd("scale", g, None, alpha=alpha)[0], f"scale bwd {alpha}")
    y = base.cuda()
    zr.zr_unary_fwd("scale", y, alpha=0.5, out=y)
    bitexact(y.cpu().numpy(), oracle.unary_fwd("scale", base, alpha=0.5), "scale in place")
    out_store = torch.empty((300, 257), device="cuda")
    zr.zr_unary_fwd("scale", to_gpu(x), alpha=2.0, out=out_store.t())
    bitexact(out_store.t().cpu().numpy(), oracle.unary_fwd("scale", x, alpha=2.0), "scale strided out")


def test_gelu_forward_and_backward():
    rng = np.random.default_rng(41)
    xs = [rng.standard_normal((64, 1031)).astype(np.float32) * 3,
          np.linspace(-14, 14, 8001, dtype=np.float32),
          np.array([0.0, -0.0, 1e-40, -1e-40, 1e-20, -0.7518, 88.0, -88.0, float("inf"),
                    -float("inf"), float("nan")], np.float32)]
    for x in xs:
        xt = torch.from_numpy(x)
        ref = oracle.unary_fwd("gelu", xt)
        got = zr.zr_unary_fwd("gelu", xt.cuda()).cpu().numpy()
        with np.errstate(all="ignore"):
            _gelu_close(got, ref, x, np.abs(ref.astype(np.float64)), f"gelu fwd {x.shape}")
        g = rng.standard_normal(x.shape).astype(np.float32)
        gref, mag = oracle.unary_bwd("gelu", g, x)
        ggot = zr.zr_unary_bwd("gelu", torch.from_numpy(g).cuda(), xt.cuda()).cpu().numpy()
        with np.errstate(all="ignore"):
            _gelu_close(ggot, gref, x, mag, f"gelu bwd {x.shape}")


def test_gelu_strided_views():
    rng = np.random.default_rng(42)
    base = torch.from_numpy((rng.standard_normal((96, 33, 2)) * 2).astype(np.float32))
    x = base[:, :, 1].t()  # [33, 96], strides (2, 66)
    ref = oracle.unary_fwd("gelu", x)
    got = zr.zr_unary_fwd("gelu", to_gpu(x)).cpu().numpy()
    _gelu_close(got, ref, x.numpy(), np.abs(ref.astype(np.float64)), "gelu fwd strided")
    g = torch.from_numpy(rng.standard_normal((33, 96)).astype(np.float32))
    gref, mag = oracle.unary_bwd("gelu", g, x)
    gx_store = torch.zeros((96, 33), device="cuda")
    zr.zr_unary_bwd("gelu", g.cuda(), to_gpu(x), grad_x=gx_store.t())
    _gelu_close(gx_store.t().cpu().numpy(), gref, x.numpy(), mag, "gelu bwd strided")


def test_unary_workload_full_sampled():
    """The benchmark's FFN-sized workload [16384, 3072], sampled."""
    host = workloads.make_inputs("u1")
    x, g = host["x"], host["g"]
    rng = np.random.default_rng(43)
    idx = np.unique(rng.integers(0, x.numel(), 20000)).astype(np.int64)
    xf = x.reshape(-1).numpy()[idx]
    gf = g.reshape(-1).numpy()[idx]
    got = zr.zr_unary_fwd("gelu", x.cuda()).reshape(-1).cpu().numpy()[idx]
    _gelu_close(got, oracle.unary_fwd("gelu", xf), xf, np.abs(oracle.unary_fwd("gelu", xf).astype(np.float64)),
                "u1 gelu fwd (sampled)")
    gx = zr.zr_unary_bwd("gelu", g.cuda(), x.cuda()).reshape(-1).cpu().numpy()[idx]
    gref, mag = oracle.unary_bwd("gelu", gf, xf)
    _gelu_close(gx, gref, xf, mag, "u1 gelu bwd (sampled)")
    s = zr.zr_unary_fwd("scale", x.cuda(), alpha=0.125).reshape(-1).cpu().numpy()[idx]
    bitexact(s, oracle.unary_fwd("scale", xf, alpha=0.125), "u1 scale fwd (sampled)")
