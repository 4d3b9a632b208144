"""GPU test of zr_binary_bwd_noalloc, the backward entry point for callers
that cannot give the library a workspace (its partial sums live in a fixed
array inside the library instead).

It is called through the C ABI twice in a row, on two problems whose plans
lay their partial sums out differently in the array (the two-gradient pass
with its grad_a and grad_b slots, then a column sum over partial slots), so
the second call runs on scratch the first one left behind.  Each result is
checked against the CPU oracle with the tolerance the parity tests use:
bit-identical where a gradient is one IEEE operation, else within
1e-5 * sum|terms| per element.  The same call through zr_binary_bwd (caller
workspace, same plan) must give the same bits.  The size limit is pinned from
both sides: a problem needing just under the array's size runs and is
correct, one needing just over is refused before anything runs.  This file is
collected last so that a stop at the first failure has already run every
other test; it also passes on its own.
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
    lib.zr_test_describe_bwd.argtypes = [ctypes.c_int, zr.ZrTensor, zr.ZrTensor, zr.ZrTensor,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                         ctypes.c_size_t]
    return lib


def _descs(g, a, b, shape_a=None, shape_b=None):
    dg, kg = zr._desc(g)
    da, ka = zr._desc(a, shape_a)
    db, kb = zr._desc(b, shape_b)
    return (dg, da, db), (kg, ka, kb)


def _plan(L, op, g, a, b, ga, gb, shape_a=None, shape_b=None):
    """The plan both backward entry points launch for these arguments."""
    (dg, da, db), keep = _descs(g, a, b, shape_a, shape_b)
    buf = ctypes.create_string_buffer(16384)
    rc = L.zr_test_describe_bwd(zr.OPS[op], dg, da, db, ga.data_ptr(), gb.data_ptr(), buf,
                                len(buf))
    assert rc == 0, L.zr_status_string(rc)
    return json.loads(buf.value)


def _noalloc(L, op, g, a, b, ga, gb, shape_a=None, shape_b=None):
    (dg, da, db), keep = _descs(g, a, b, shape_a, shape_b)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.zr_binary_bwd_noalloc(zr.OPS[op], dg, da, db, ga.data_ptr(), gb.data_ptr(), stream)


def _check_vs_oracle(op, host_g, host_a, host_b, got):
    ref_a, ref_b, sa, sb = oracle.binary_bwd(op, host_g, host_a, host_b)
    n_out = host_g.numel()
    for which, x, r, s in ((0, got[0], ref_a, sa), (1, got[1], ref_b, sb)):
        x = x.cpu().numpy()
        what = f"noalloc {op} grad_{'ab'[which]}"
        if x.size == n_out and not (op == "div" and which == 1):
            bitexact(x, r, what)
        else:
            within(x, r, s, what)


def test_noalloc_matches_oracle_twice_on_shared_scratch(L):
    # First call: 8-d div with both gradients reduced, the two-gradient pass
    # (grad_a's and grad_b's partial slots in the scratch; it needs a
    # 16-byte-vector inner dim and enough steps, hence these sizes).
    h1 = workloads.make_inputs("c5b", a=(2, 1, 4, 1, 8, 1, 16, 32), b=(1, 3, 1, 5, 1, 6, 1, 32))
    # Second call: bias-add backward, a column sum over many rows; rows of
    # 1030 floats rule out 16-byte vectors (and with them the cluster plan
    # that needs no partials), so the sum goes through partial slots in the
    # scratch with another layout.
    h2 = workloads.make_inputs("c2", R=4096, C=1030)
    cases = [("div", h1["g"], h1["a"], h1["b"], "sab"), ("add", h2["g"], h2["x"], h2["bias"], "reduce")]
    plans = []
    for op, g, a, b, kernel in cases:
        dg, da, db = to_gpu(g), to_gpu(a), to_gpu(b)
        ga = torch.full(a.shape, float("nan"), device="cuda")
        gb = torch.full(b.shape, float("nan"), device="cuda")
        plan = _plan(L, op, dg, da, db, ga, gb)
        assert 0 < plan["ws_run"] <= SCRATCH_BYTES, plan
        assert plan["plans"][0]["kernel"] == kernel, plan
        if kernel == "reduce":
            assert plan["plans"][0]["nslots"] > 1 and plan["plans"][0]["cluster"] == 1, plan
        plans.append(plan)
        rc = _noalloc(L, op, dg, da, db, ga, gb)
        assert rc == 0, L.zr_status_string(rc)
        torch.cuda.synchronize()
        _check_vs_oracle(op, g, a, b, (ga, gb))
        # The workspace entry point runs the same plan, so the same bits.
        ref = zr.zr_binary_bwd(op, dg, da, db)
        torch.cuda.synchronize()
        for x, r, w in ((ga, ref[0], "a"), (gb, ref[1], "b")):
            bitexact(x.cpu().numpy(), r.cpu().numpy(), f"noalloc vs workspace {op} grad_{w}")
    assert plans[0]["plans"][0]["kernel"] != plans[1]["plans"][0]["kernel"]


def test_noalloc_runs_just_under_the_limit(L):
    # [16384, 16383] + [16383] add: 128 partial slots of 16383 floats, 512
    # bytes short of the array's size.  x is not read by add's backward.
    R, C = 16384, 16383
    gen = torch.Generator().manual_seed(1010)
    host_g = torch.randn((R, C), generator=gen, dtype=torch.float32)
    g = host_g.cuda()
    ga = torch.full((R, C), float("nan"), device="cuda")
    gb = torch.full((C,), float("nan"), device="cuda")
    plan = _plan(L, "add", g, None, None, ga, gb, shape_a=(R, C), shape_b=(C,))
    assert SCRATCH_BYTES - 4096 < plan["ws_run"] <= SCRATCH_BYTES, plan
    rc = _noalloc(L, "add", g, None, None, ga, gb, shape_a=(R, C), shape_b=(C,))
    assert rc == 0, L.zr_status_string(rc)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    cols = np.concatenate([[0, 1, C - 2, C - 1], rng.choice(C, 60, replace=False)])
    vals, sabs = oracle.binary_bwd_at("add", 1, host_g, None, None, cols, shape_a=(R, C),
                                      shape_b=(C,))
    within(gb.cpu().numpy()[cols], vals, sabs, "noalloc add grad_b near the limit")
    idx = np.concatenate([[0, R * C - 1], rng.choice(R * C, 4000, replace=False)])
    vals, _ = oracle.binary_bwd_at("add", 0, host_g, None, None, idx, shape_a=(R, C),
                                   shape_b=(C,))
    bitexact(ga.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy(), vals,
             "noalloc add grad_a near the limit")


def test_noalloc_rejects_problems_just_beyond_the_scratch(L):
    # [32768, 8417] + [8417] add: 256 partial slots of 8417 floats, 230,400
    # bytes more than the array holds.
    R, C = 32768, 8417
    g = torch.zeros((R, C), device="cuda")
    ga = torch.empty((R, C), device="cuda")
    gb = torch.full((C,), 7.0, device="cuda")
    plan = _plan(L, "add", g, None, None, ga, gb, shape_a=(R, C), shape_b=(C,))
    assert SCRATCH_BYTES < plan["ws_run"] <= SCRATCH_BYTES + (1 << 20), plan
    rc = _noalloc(L, "add", g, None, None, ga, gb, shape_a=(R, C), shape_b=(C,))
    assert rc == ZR_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(gb == 7.0)  # nothing ran
