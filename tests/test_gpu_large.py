"""Sizes past 32-bit indexing: a [65537, 32768] float32 operand
(2,147,516,416 elements, 8.6 GB, element offsets above 2^31 and byte offsets
above 2^33) with a [32768] bias, forward and backward through the C ABI; and
bfloat16 GeLU by table on an operand of the same shape.
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


def test_bf16_gelu_table_past_32_bit_offsets():
    """bfloat16 GeLU forward and backward on a [65537, 32768] operand
    (element offsets past 2^31) through the table kernel: sampled elements,
    the first and the last, equal bit for bit the arithmetic path's results
    on the same values (a small call, below the table's size)."""
    gen = torch.Generator(device="cuda").manual_seed(1802)
    x = (torch.randn((R, C), generator=gen, device="cuda") * 2).to(torch.bfloat16)
    g = torch.randn((R, C), generator=gen, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(1803)
    flat_idx = np.concatenate([[0, 1, R * C - 2, R * C - 1], rng.integers(0, R * C, 4000)])
    idx = torch.from_numpy(flat_idx.astype(np.int64)).cuda()
    xs, gs = x.reshape(-1)[idx].contiguous(), g.reshape(-1)[idx].contiguous()
    y = zr.zr_unary_fwd("gelu", x)
    got_f = y.reshape(-1)[idx]
    del y
    gx = zr.zr_unary_bwd("gelu", g, x)
    got_b = gx.reshape(-1)[idx]
    del gx
    ref_f = zr.zr_unary_fwd("gelu", xs)
    ref_b = zr.zr_unary_bwd("gelu", gs, xs)
    torch.cuda.synchronize()
    for got, ref, what in ((got_f, ref_f, "forward"), (got_b, ref_b, "backward")):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), \
            f"bf16 GeLU {what} past 2^31 elements"
