"""GPU parity of zr_binary_bwd_ex: gradients written into strided layouts
and accumulated into existing values (grad += result), through the C ABI,
against the oracle's gradients and its AccumulateGrad addition.

Acceptance: a gradient that is one binary32 operation (and, accumulated, one
more binary32 addition) is bit-identical; a summed gradient is within
1e-5 * (sum|terms| + |old value|) per element.  Every backward plan family
is covered: elementwise (no reduction), one reduced gradient on partial
slots, on thread-block clusters and with the inner dim reduced, both reduced
(the fused one-pass kernel) and a full sum.  Elements around a strided view
stay untouched.
"""
import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
from parity import bitexact, within

pytestmark = pytest.mark.gpu

OPS = ["add", "sub", "mul", "div"]

# (a shape, b shape): elementwise; slots (ragged rows rule out 16-byte
# vectors); cluster; inner dim reduced; both reduced (fused pass); full sum.
LAYOUTS = [((33, 65), (33, 65)), ((517, 1030), (1030,)), ((2048, 1024), (1024,)),
           ((5, 67, 203), (1, 67, 1)), ((2, 1, 256, 4), (1, 3, 1, 4)), ((64, 64), (1,))]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


def _strided(shape, rng, kind):
    """A device view of `shape` that is not dense row-major, inside a larger
    buffer filled with a sentinel; returns (view, buffer, mask of the view's
    elements within the buffer)."""
    if kind == "step":
        buf = torch.full((*shape, 2), 7.25, device="cuda")
        view = buf[..., 0]
    else:  # reversed dims (a transpose for 2-d)
        buf = torch.full(tuple(reversed(shape)), 7.25, device="cuda")
        view = buf.permute(*reversed(range(len(shape))))
    mark = torch.zeros_like(buf)
    mark_view = mark[..., 0] if kind == "step" else mark.permute(*reversed(range(len(shape))))
    mark_view.fill_(1.0)
    old = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
    view.copy_(old.cuda())
    return view, buf, mark.bool(), old


def _expect(op, which, n_out, got, ref, sabs, old, acc, what):
    reduced = ref.size != n_out
    single = not reduced and not (op == "div" and which == 1)
    want = oracle.accumulate(old, ref) if acc else ref
    if single:
        bitexact(got, want, what)
    else:
        bound = sabs + (np.abs(old.astype(np.float64)) if acc else 0.0)
        within(got, want, bound, what)


@pytest.mark.parametrize("op", OPS)
def test_accumulate_and_strided_gradients(op):
    rng = np.random.default_rng(1200 + OPS.index(op))
    for sa, sb in LAYOUTS:
        a = torch.from_numpy(rng.standard_normal(sa).astype(np.float32))
        b = torch.from_numpy((np.sign(rng.standard_normal(sb)) * (0.5 + rng.random(sb))).astype(np.float32))
        g = torch.from_numpy(rng.standard_normal(np.broadcast_shapes(sa, sb)).astype(np.float32))
        ra, rb, s1, s2 = oracle.binary_bwd(op, g, a, b)
        n_out = g.numel()
        ad, bd, gd = a.cuda(), b.cuda(), g.cuda()
        for mode in ("dense_acc", "strided", "strided_acc", "mixed"):
            acc = (mode in ("dense_acc", "strided_acc", "mixed"), mode in ("dense_acc", "strided_acc"))
            grads, checks = [], []
            for w, shape in enumerate((sa, sb)):
                strided = mode in ("strided", "strided_acc") or (mode == "mixed" and w == 1)
                if strided:
                    view, buf, mark, old = _strided(shape, rng, "step" if w == 0 else "reverse")
                else:
                    old = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
                    view, buf, mark = old.cuda(), None, None
                grads.append(view)
                checks.append((buf, mark, old.numpy()))
            zr.zr_binary_bwd_ex(op, gd, ad, bd, grad_a=grads[0], grad_b=grads[1], accumulate=acc)
            torch.cuda.synchronize()
            for w, (ref, sabs) in enumerate(((ra, s1), (rb, s2))):
                buf, mark, old = checks[w]
                what = f"bwd_ex {op} {sa} {sb} {mode} grad_{'ab'[w]}"
                _expect(op, w, n_out, grads[w].cpu().numpy(), ref, sabs, old, acc[w], what)
                if buf is not None:
                    assert torch.all(buf[~mark] == 7.25), f"{what}: wrote outside the view"


def test_accumulate_twice_and_empty():
    """Two accumulating calls add two gradients; with grad_out empty an
    accumulated gradient keeps its values and a written one becomes zero."""
    rng = np.random.default_rng(1300)
    g = torch.from_numpy(rng.standard_normal((512, 1024)).astype(np.float32))
    x = torch.from_numpy(rng.standard_normal((512, 1024)).astype(np.float32))
    w = torch.from_numpy(rng.standard_normal((1024,)).astype(np.float32))
    gx, gw, _, sw = oracle.binary_bwd("mul", g, x, w)
    acc_x = torch.zeros((512, 1024), device="cuda")
    acc_w = torch.zeros((1024,), device="cuda")
    for _ in range(2):
        zr.zr_binary_bwd_ex("mul", g.cuda(), x.cuda(), w.cuda(), grad_a=acc_x, grad_b=acc_w,
                            accumulate=(True, True))
    want_x = oracle.accumulate(oracle.accumulate(np.zeros_like(gx), gx), gx)
    bitexact(acc_x.cpu().numpy(), want_x, "twice grad_x")
    within(acc_w.cpu().numpy(), 2 * gw.astype(np.float64), 2 * sw, "twice grad_w")
    ge = torch.empty((0, 1024), device="cuda")
    xe = torch.empty((0, 1024), device="cuda")
    keep = torch.full((1024,), 3.5, device="cuda")
    zero = torch.full((1024,), 3.5, device="cuda")
    zr.zr_binary_bwd_ex("mul", ge, xe, w.cuda(), grad_b=keep, accumulate=(False, True))
    zr.zr_binary_bwd_ex("mul", ge, xe, w.cuda(), grad_b=zero, accumulate=(False, False))
    assert torch.all(keep == 3.5) and torch.all(zero == 0.0)
