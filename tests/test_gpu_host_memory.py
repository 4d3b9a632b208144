"""Operands in pinned host memory through the C ABI: the device addresses a
page-locked buffer at the same pointer, so the kernels read inputs from (and
write outputs to) host memory directly.  Results are bit-identical to the
oracle's forward; pageable host memory is refused on the host before any
launch (ZR_ERR_DEVICE)."""
import ctypes

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
from parity import bitexact

pytestmark = pytest.mark.gpu

ZR_ERR_DEVICE = -6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


def _raw(t):
    """zr_tensor for any torch tensor (the binding itself takes CUDA tensors only)."""
    sizes, strides = zr._i64(t.shape), zr._i64(t.stride())
    return zr.ZrTensor(t.data_ptr(), t.dim(), sizes, strides), (sizes, strides)


def _fwd(op, a, b, out):
    da, ka = _raw(a)
    db, kb = _raw(b)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return zr.lib().zr_binary_fwd(zr.OPS[op], da, db, ctypes.c_void_p(out.data_ptr()), None, st)


@pytest.mark.parametrize("op", ["add", "div"])
def test_pinned_host_operands(op):
    rng = np.random.default_rng(1400)
    a = torch.from_numpy(rng.standard_normal((1030, 1024)).astype(np.float32))
    b = torch.from_numpy((0.5 + rng.random(1024)).astype(np.float32))
    want = oracle.binary_fwd(op, a, b)
    ha, hb = a.pin_memory(), b.pin_memory()
    da, db = a.cuda(), b.cuda()
    for name, x, y, on_host in (("host a", ha, db, False), ("host b", da, hb, False),
                                ("host out", da, db, True), ("all host", ha, hb, True)):
        out = (torch.empty((1030, 1024)).pin_memory() if on_host
               else torch.empty((1030, 1024), device="cuda"))
        assert _fwd(op, x, y, out) == 0, name
        torch.cuda.synchronize()
        bitexact(out.cpu().numpy(), want, f"{op} {name}")


def test_pageable_host_memory_is_refused():
    a = torch.ones((64, 64))  # pageable
    b = torch.ones((64,), device="cuda")
    out = torch.full((64, 64), 5.0, device="cuda")
    assert _fwd("add", a, b, out) == ZR_ERR_DEVICE
    torch.cuda.synchronize()
    assert torch.all(out == 5.0)
