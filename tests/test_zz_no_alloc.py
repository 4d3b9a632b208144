"""GPU test of zr_binary_bwd_noalloc, the backward entry point for callers
that cannot give the library a workspace (its partial sums live in a fixed
array inside the library instead).

It is called through the C ABI twice in a row, on two different problems,
so the second call runs on scratch the first one left behind; each result
must match zr_binary_bwd (the entry point that takes a caller workspace)
within the tolerance the parity tests use: bit-identical where a gradient is
one IEEE operation, else 1e-5 * sum|terms| per element (sums from the
oracle).  A problem too large for the fixed array must be refused before
anything runs.  This file is collected last so that a stop at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads
from parity import bitexact, to_gpu, within

pytestmark = pytest.mark.gpu

ZR_ERR_WORKSPACE = -7
SCRATCH_BYTES = 8 << 20  # ZR_STATIC_SCRATCH_BYTES in include/zr.h


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    lib = zr.lib()
    lib.zr_binary_bwd_noalloc.argtypes = [ctypes.c_int, zr.ZrTensor, zr.ZrTensor, zr.ZrTensor,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.zr_binary_bwd_noalloc.restype = ctypes.c_int
    return lib


def _noalloc(L, op, g, a, b):
    ga = torch.full(a.shape, float("nan"), device="cuda")
    gb = torch.full(b.shape, float("nan"), device="cuda")
    dg, kg = zr._desc(g)
    da, ka = zr._desc(a)
    db, kb = zr._desc(b)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.zr_binary_bwd_noalloc(zr.OPS[op], dg, da, db, ga.data_ptr(), gb.data_ptr(), stream)
    assert rc == 0, L.zr_status_string(rc)
    torch.cuda.synchronize()
    return ga, gb


def _check(op, host_g, host_a, host_b, got, ref):
    _, _, sa, sb = oracle.binary_bwd(op, host_g, host_a, host_b)
    n_out = host_g.numel()
    for which, x, r, s in ((0, got[0], ref[0], sa), (1, got[1], ref[1], sb)):
        x, r = x.cpu().numpy(), r.cpu().numpy()
        single_op = x.size == n_out and not (op == "div" and which == 1)
        if single_op:
            bitexact(x, r, f"noalloc {op} grad_{'ab'[which]}")
        else:
            within(x, r, s, f"noalloc {op} grad_{'ab'[which]}")


def test_noalloc_matches_workspace_entry_point_twice(L):
    # First call: 8-d div with both gradients reduced (uses the scratch).
    h1 = workloads.make_inputs("c5b", **workloads.small_dims("c5b"))
    # Second call: bias-add backward, a column sum over many rows; rows of
    # 1030 floats rule out 16-byte vectors, so the sum goes through partial
    # slots in the scratch too, with a different layout of partials.
    h2 = workloads.make_inputs("c2", R=4096, C=1030)
    cases = [("div", h1["g"], h1["a"], h1["b"]), ("add", h2["g"], h2["x"], h2["bias"])]
    for op, g, a, b in cases:
        dg, da, db = to_gpu(g), to_gpu(a), to_gpu(b)
        ref = zr.zr_binary_bwd(op, dg, da, db)
        torch.cuda.synchronize()
        got = _noalloc(L, op, dg, da, db)
        _check(op, g, a, b, got, ref)


def test_noalloc_rejects_problems_beyond_the_scratch(L):
    # [8192, 65535] + [65535]: the column sum's partials (64 slots of 65535
    # floats) need more than the fixed array holds.
    g = torch.zeros((8192, 65535), device="cuda")
    x = torch.zeros((8192, 65535), device="cuda")
    bias = torch.zeros((65535,), device="cuda")
    need = ctypes.c_size_t(0)
    dg, kg = zr._desc(g)
    dx, kx = zr._desc(x)
    db, kb = zr._desc(bias)
    ga = torch.empty_like(x)
    gb = torch.empty_like(bias)
    assert zr.lib().zr_binary_bwd(0, dg, dx, db, ga.data_ptr(), gb.data_ptr(), None,
                                  ctypes.byref(need), None) == 0
    assert need.value > SCRATCH_BYTES
    gb.fill_(7.0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.zr_binary_bwd_noalloc(0, dg, dx, db, ga.data_ptr(), gb.data_ptr(), stream)
    assert rc == ZR_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(gb == 7.0)  # nothing ran
