"""Sizes past 32-bit indexing: a [65537, 32768] float32 operand
(2,147,516,416 elements, 8.6 GB, element offsets above 2^31 and byte offsets
above 2^33) with a [32768] bias, forward and backward through the C ABI.
Inputs are drawn on the device from a seeded generator; the oracle evaluates
sampled outputs, and full column sums for sampled columns, from those inputs
copied back."""
import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
from parity import bitexact, within

pytestmark = pytest.mark.gpu

R, C = 65537, 32768


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * 2**30:
        pytest.skip("needs about 30 GB of free device memory")
    zr.build()
    zr.lib()


def test_past_32_bit_offsets_forward_and_backward():
    gen = torch.Generator(device="cuda").manual_seed(1800)
    a = torch.randn((R, C), generator=gen, device="cuda")
    b = torch.randn((C,), generator=gen, device="cuda")
    assert a.numel() > 2**31
    rng = np.random.default_rng(1801)
    rows = np.concatenate([[0, R // 2, R - 2, R - 1], rng.integers(0, R, 60)])
    cols = np.concatenate([[0, C - 1], rng.integers(0, C, 62)])
    ri, ci = (torch.from_numpy(x.astype(np.int64)).cuda() for x in np.meshgrid(rows, cols, indexing="ij"))
    a_s = a[ri, ci].cpu()
    b_s = b[ci].cpu()

    out = zr.zr_binary_fwd("mul", a, b)
    got = out[ri, ci].cpu().numpy()
    del out
    bitexact(got, oracle.binary_fwd("mul", a_s.reshape(-1), b_s.reshape(-1)).reshape(got.shape),
             "mul forward past 2^31 elements")

    # Backward of mul with grad_out = a: grad_a = a * b densely, grad_b[j] = sum_i a[i, j]^2.
    ga, gb = zr.zr_binary_bwd("mul", a, a, b)
    torch.cuda.synchronize()
    got_a = ga[ri, ci].cpu().numpy()
    del ga
    bitexact(got_a, oracle.binary_fwd("mul", a_s.reshape(-1), b_s.reshape(-1)).reshape(got_a.shape),
             "mul grad_a past 2^31 elements")
    sample_cols = np.unique(cols)[:16]
    for j in sample_cols:
        col = a[:, int(j)].cpu()
        # sum_i a_ij * a_ij: the oracle's backward of mul on one column.
        ra, rb, sa, sb = oracle.binary_bwd("mul", col.view(R, 1), col.view(R, 1), b[int(j)].cpu().view(1))
        within(gb[int(j)].cpu().numpy().reshape(1), rb.reshape(1), sb.reshape(1),
               f"grad_b column {j}")
