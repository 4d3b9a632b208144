"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs, through the C ABI (Python binding).  Needs a CUDA GPU (GB300).

* every workload at reduced sizes with the same structure (several tiles and
  ragged tails), compared element by element;
* every workload at its full size, in the launch configuration the benchmark
  uses, compared on sampled outputs the oracle computes one by one;
* random shapes, strides, ops and views; edge cases (empty, scalar, rank 8,
  special values, misaligned and in-place buffers, strided outputs);
* bitwise run-to-run determinism and host-side error reporting.
"""
import ctypes
import json

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads
from parity import (bitexact, compare_workload, is_single_op_grad, run_gpu, run_oracle, to_gpu,
                    within)

pytestmark = pytest.mark.gpu

OPS = ["add", "sub", "mul", "div"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


# ----------------------------------------------------------- workloads, small sizes

@pytest.mark.parametrize("name", workloads.NAMES)
def test_workload_small(name):
    host = workloads.make_inputs(name, **workloads.small_dims(name))
    gpu = run_gpu(name, host)
    ref, sums = run_oracle(name, host)
    compare_workload(name, host, gpu, ref, sums)


@pytest.mark.parametrize("name", workloads.NAMES)
def test_workload_small_other_seed(name):
    host = workloads.make_inputs(name, seed=77, **workloads.small_dims(name))
    gpu = run_gpu(name, host)
    ref, sums = run_oracle(name, host)
    compare_workload(name, host, gpu, ref, sums)


# ----------------------------------------------------------- workloads, full sizes

def _sample(n, k, rng):
    idx = rng.integers(0, n, k)
    return np.unique(np.concatenate([idx, [0, n - 1, n // 2]]).astype(np.int64))


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_workload_full_exhaustive(name):
    host = workloads.make_inputs(name)
    gpu = run_gpu(name, host)
    ref, sums = run_oracle(name, host)
    compare_workload(name, host, gpu, ref, sums)


@pytest.mark.parametrize("name", ["c3", "c4", "c5a", "c5b"])
def test_workload_full_sampled(name):
    """Full-size inputs; the oracle evaluates sampled outputs of every step
    from its own intermediates (never the GPU's)."""
    rng = np.random.default_rng(5)
    host = workloads.make_inputs(name)
    gpu = run_gpu(name, host)
    env = dict(host)  # oracle-side values of every tensor named in the steps
    steps = workloads.STEPS[name]
    last_fwd = max(i for i, s in enumerate(steps) if s[0] == "fwd")
    for i, step in enumerate(steps):
        if step[0] == "fwd":
            _, op, an, bn, on = step
            n = gpu[on].numel()
            idx = _sample(n, 4000, rng)
            vals = oracle.binary_fwd_at(op, env[an], env[bn], idx)
            bitexact(gpu[on].reshape(-1).numpy()[idx], vals, f"{name} fwd {on} (sampled)")
            # Later steps read this intermediate: the oracle makes its own.
            if i < last_fwd or any(on in s[2:5] for s in steps[i + 1:] if s[0] == "bwd"):
                env[on] = torch.from_numpy(oracle.binary_fwd(op, env[an], env[bn]))
        else:
            _, op, gn, an, bn, gan, gbn = step
            out_numel = env[gn].numel()
            for which, gname, src in ((0, gan, an), (1, gbn, bn)):
                n = gpu[gname].numel()
                idx = _sample(n, 400 if n > out_numel // 64 else 2000, rng)
                if n <= 64:
                    idx = np.arange(n, dtype=np.int64)
                vals, sabs = oracle.binary_bwd_at(op, which, env[gn], env[an], env[bn], idx)
                got = gpu[gname].reshape(-1).numpy()[idx]
                reduced = n != out_numel
                what = f"{name} bwd {op} -> {gname} (sampled)"
                if not reduced and not (op == "div" and which == 1):
                    bitexact(got, vals, what)
                else:
                    within(got, vals, sabs, what)
            used_later = any(gan in s[2:5] for s in steps[i + 1:])
            if used_later:
                ga, _, _, _ = oracle.binary_bwd(op, env[gn], env[an], env[bn], want_b=False)
                env[gan] = torch.from_numpy(ga)


# ----------------------------------------------------------- random fuzz

def _rand_view(rng, shape, kind=None):
    kind = rng.integers(0, 4) if kind is None else kind
    if kind == 0 or len(shape) == 0:
        return torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
    if kind == 1:
        perm = rng.permutation(len(shape))
        base = torch.from_numpy(rng.standard_normal([shape[p] for p in perm]).astype(np.float32))
        return base.permute(*np.argsort(perm).tolist())
    if kind == 2:
        big = torch.from_numpy(rng.standard_normal([2 * s + 1 for s in shape]).astype(np.float32))
        return big[tuple(slice(0, 2 * s, 2) for s in shape)]
    flat = torch.from_numpy(rng.standard_normal(int(np.prod(shape)) + 1).astype(np.float32))
    return flat[1:].view(shape)  # misaligned by one element


def _rand_pair(rng):
    n = int(rng.integers(0, 7))
    out = [int(v) for v in rng.choice([1, 2, 3, 4, 5, 7, 8, 16, 33], n)]
    sa = [s if rng.random() < 0.6 else 1 for s in out]
    sb = [s if rng.random() < 0.6 else 1 for s in out]
    sa = sa[int(rng.integers(0, n + 1)) if n else 0:]
    sb = sb[int(rng.integers(0, n + 1)) if n else 0:]
    return tuple(sa), tuple(sb)


def _b_for(op, t, rng):
    if op == "div":
        sign = torch.from_numpy(np.where(rng.random(tuple(t.shape)) < 0.5, -1.0, 1.0).astype(np.float32))
        return t.abs() + 0.5 * sign.sign()
    return t


@pytest.mark.parametrize("seed", range(4))
def test_random_fwd_bwd(seed):
    rng = np.random.default_rng(1000 + seed)
    for it in range(60):
        sa, sb = _rand_pair(rng)
        op = OPS[it % 4]
        a = _rand_view(rng, sa)
        b = _rand_view(rng, sb)
        if op == "div":
            b = (b.abs() + 0.5) * torch.from_numpy(
                np.where(rng.random(sb) < 0.5, -1.0, 1.0).astype(np.float32)).reshape(sb)
            b = b if rng.random() < 0.5 else _rand_like_view(rng, b)
        out = zr.zr_binary_fwd(op, to_gpu(a), to_gpu(b)).cpu().numpy()
        bitexact(out, oracle.binary_fwd(op, a, b), f"fwd {op} {sa} {sb}")
        out_shape = np.broadcast_shapes(sa, sb)
        g = _rand_view(rng, out_shape)
        want_a, want_b = [(True, True), (True, False), (False, True)][it % 3]
        ga, gb = zr.zr_binary_bwd(op, to_gpu(g), to_gpu(a), to_gpu(b), want_a=want_a, want_b=want_b)
        ra, rb, sa_abs, sb_abs = oracle.binary_bwd(op, g, a, b, want_a=want_a, want_b=want_b)
        n_out = int(np.prod(out_shape))
        for which, x, r, s, shp in ((0, ga, ra, sa_abs, sa), (1, gb, rb, sb_abs, sb)):
            if x is None:
                assert r is None
                continue
            x = x.cpu().numpy()
            reduced = int(np.prod(shp)) != n_out
            what = f"bwd {op} grad_{'ab'[which]} {sa} {sb}"
            if not reduced and not (op == "div" and which == 1):
                bitexact(x, r, what)
            else:
                within(x, r, s, what)


def _rand_like_view(rng, t):
    """Same values, stored transposed/stepped (keeps the logical tensor)."""
    if t.dim() < 2:
        return t
    return t.t().contiguous().t() if t.dim() == 2 else t.permute(*reversed(range(t.dim()))).contiguous().permute(*reversed(range(t.dim())))


@pytest.mark.parametrize("seed", range(3))
def test_random_sum_to_shape(seed):
    rng = np.random.default_rng(2000 + seed)
    for it in range(60):
        n = int(rng.integers(0, 7))
        shape = tuple(int(v) for v in rng.choice([1, 2, 3, 5, 8, 16, 31, 64], n))
        target = [s if rng.random() < 0.5 else 1 for s in shape]
        target = tuple(target[int(rng.integers(0, n + 1)) if n else 0:])
        x = _rand_view(rng, shape)
        got = zr.zr_sum_to_shape(to_gpu(x), target).cpu().numpy()
        ref, sabs = oracle.sum_to_shape(x, target)
        if int(np.prod(target)) == x.numel():
            bitexact(got, ref, f"sum_to_shape copy {shape}->{target}")
        else:
            within(got, ref, sabs, f"sum_to_shape {shape}->{target}")


def test_sum_to_shape_large_reductions():
    rng = np.random.default_rng(3)
    # The last two: many outputs (second pass with 4 outputs per thread) and
    # a ragged count of them (one per thread).
    cases = [((4096, 1024), (1024,)), ((4096, 1024), (4096, 1)), ((64, 64, 64, 64), (1,)),
             ((3, 1000, 7, 33), (1000, 1, 1)), ((1 << 20) + 3,), ((700, 20000), (20000,)),
             ((1500, 10001), (10001,))]
    for case in cases:
        shape, target = (case if len(case) == 2 else (case[0], (1,)))
        x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
        got = zr.zr_sum_to_shape(x.cuda(), target).cpu().numpy()
        ref, sabs = oracle.sum_to_shape(x, target)
        within(got, ref, sabs, f"sum_to_shape {shape}->{target}")


def test_adversarial_all_positive_sums():
    """Long all-positive sums, where a plain fp32 chain would drift most."""
    x = torch.full((1 << 24,), 0.1, dtype=torch.float32) + torch.rand(1 << 24, generator=torch.Generator().manual_seed(1))
    got = zr.zr_sum_to_shape(x.cuda(), (1,)).cpu().numpy()
    ref, sabs = oracle.sum_to_shape(x, (1,))
    within(got, ref, sabs, "sum of 2^24 positives", tol=1e-6)
    g = torch.rand((16384, 768), generator=torch.Generator().manual_seed(2)) + 1.0
    bias = torch.zeros(768)
    _, gb = zr.zr_binary_bwd("add", g.cuda(), None, bias.cuda(), want_a=False, shape_a=(16384, 768))
    ref = oracle.sum_to_shape(g, (768,))
    within(gb.cpu().numpy(), ref[0], ref[1], "column sums of positives", tol=1e-6)


# ----------------------------------------------------------- edge cases

def test_special_values_bit_exact():
    sp = torch.tensor([0.0, -0.0, 1.0, -1.0, float("inf"), -float("inf"), float("nan"), 1e-45,
                       -1e-45, 1.17e-38, 3.4e38, -3.4e38, 8.0, 0.125, 1e-30, 7.0], dtype=torch.float32)
    a = sp.view(-1, 1).expand(16, 16).contiguous()
    b = sp.view(1, -1).expand(16, 16).contiguous()
    for op in OPS:
        for x, y in ((a, b), (sp.view(-1, 1), sp.view(1, -1))):
            out = zr.zr_binary_fwd(op, x.cuda(), y.cuda()).cpu().numpy()
            bitexact(out, oracle.binary_fwd(op, x, y), f"special fwd {op}")
        g = torch.roll(a, 3, 1).contiguous()
        ga, gb = zr.zr_binary_bwd(op, g.cuda(), a.cuda(), b.cuda())
        ra, rb, _, sb = oracle.binary_bwd(op, g, a, b)
        bitexact(ga.cpu().numpy(), ra, f"special grad_a {op}")
        if op != "div":
            bitexact(gb.cpu().numpy(), rb, f"special grad_b {op}")


def test_empty_and_scalar():
    e = torch.empty((0, 3), device="cuda")
    b = torch.ones((1, 3), device="cuda")
    out = zr.zr_binary_fwd("add", e, b)
    assert out.shape == (0, 3)
    ga, gb = zr.zr_binary_bwd("mul", torch.empty((0, 3), device="cuda"), e, b)
    assert ga.shape == (0, 3)
    assert torch.equal(gb.cpu(), torch.zeros(1, 3))
    s1 = torch.tensor(3.0).cuda()
    s2 = torch.tensor(2.0).cuda()
    assert zr.zr_binary_fwd("mul", s1, s2).item() == 6.0
    ga, gb = zr.zr_binary_bwd("mul", torch.tensor(1.0).cuda(), s1, s2)
    assert (ga.item(), gb.item()) == (2.0, 3.0)
    x = torch.randn(5, 7).cuda()
    assert torch.equal(zr.zr_sum_to_shape(torch.empty(0, 7, device="cuda"), (7,)).cpu(), torch.zeros(7))
    assert torch.equal(zr.zr_sum_to_shape(x, (5, 7)).cpu(), x.cpu())


def test_worked_gradient_on_gpu():
    """z = x*y + x at x=3, y=2: dz/dx = 3, dz/dy = 3 (Zero book, Autograd
    page, sections 链式法则 and 计算图), composed from the library's calls."""
    x = torch.tensor([3.0]).cuda()
    y = torch.tensor([2.0]).cuda()
    xy = zr.zr_binary_fwd("mul", x, y)
    z = zr.zr_binary_fwd("add", xy, x)
    assert z.item() == 9.0
    g_xy, g_x1 = zr.zr_binary_bwd("add", torch.ones(1).cuda(), xy, x)
    g_x2, g_y = zr.zr_binary_bwd("mul", g_xy, x, y)
    assert (g_x1 + g_x2).item() == 3.0 and g_y.item() == 3.0


def test_rank8_and_ragged():
    rng = np.random.default_rng(8)
    sa = (2, 1, 3, 1, 2, 1, 3, 5)
    sb = (1, 3, 1, 2, 1, 3, 1, 5)
    a = torch.from_numpy(rng.standard_normal(sa).astype(np.float32))
    b = torch.from_numpy((rng.random(sb) + 0.5).astype(np.float32))
    g = torch.from_numpy(rng.standard_normal(np.broadcast_shapes(sa, sb)).astype(np.float32))
    for op in OPS:
        bitexact(zr.zr_binary_fwd(op, a.cuda(), b.cuda()).cpu().numpy(), oracle.binary_fwd(op, a, b))
        ga, gb = zr.zr_binary_bwd(op, g.cuda(), a.cuda(), b.cuda())
        ra, rb, s1, s2 = oracle.binary_bwd(op, g, a, b)
        within(ga.cpu().numpy(), ra, s1, f"rank8 {op} grad_a")
        within(gb.cpu().numpy(), rb, s2, f"rank8 {op} grad_b")


def _fwd_kernel(op, a, b, out):
    L = zr.lib()
    L.zr_test_describe_fwd.argtypes = [ctypes.c_int, zr.ZrTensor, zr.ZrTensor, ctypes.c_void_p,
                                       ctypes.POINTER(ctypes.c_int64), ctypes.c_char_p,
                                       ctypes.c_size_t]
    da, ka = zr._desc(a)
    db, kb = zr._desc(b)
    ost = zr._i64(out.stride())
    buf = ctypes.create_string_buffer(4096)
    assert L.zr_test_describe_fwd(zr.OPS[op], da, db, out.data_ptr(), ost, buf, 4096) == 0
    import json
    return json.loads(buf.value.decode())["kernel"]


def test_transposed_input_tiles():
    """Forward with one input stored transposed (unit stride along an outer
    dim): interior 4x4 blocks with 16-byte accesses, blocks cut by ragged p
    and q edges, y broadcast along q, along p or not at all, the transposed
    input on either side of a non-commutative op, and an output whose rows
    are not 16-byte aligned (scalar path)."""
    rng = np.random.default_rng(31)
    # p = M = 130: one full p tile and a 2-wide one (a 4x4 block cut by the
    # p edge); q = Q = 203 (a block cut by the q edge).  x's storage rows are
    # padded to 136 floats so that its rows stay 16-byte aligned.
    P, M, Q = 3, 130, 203
    st = torch.from_numpy(rng.standard_normal((P, Q, 136)).astype(np.float32)).cuda()
    xt = st[:, :, :M].transpose(1, 2)  # [P, M, Q], unit stride along M
    dense = torch.from_numpy(rng.standard_normal((P, M, Q)).astype(np.float32) + 3.0).cuda()
    ys = {
        "along_p": torch.from_numpy(rng.standard_normal((1, M, 1)).astype(np.float32) + 3.0).cuda(),
        "along_q": torch.from_numpy(rng.standard_normal((1, 1, Q)).astype(np.float32) + 3.0).cuda(),
        "full": dense,
    }
    pitched = {n: torch.empty((P, M, n), device="cuda") for n in (204, 205)}
    outs = {"pitch_204": lambda: pitched[204][:, :, :Q],   # aligned rows: 16-byte stores
            "pitch_205": lambda: pitched[205][:, :, :Q],   # unaligned rows: scalar
            "dense": lambda: torch.empty((P, M, Q), device="cuda")}
    for op in OPS:
        for yname, y in ys.items():
            for xa in (True, False):
                a, b = (xt, y) if xa else (y, xt)
                for oname, mk in outs.items():
                    out = mk()
                    assert _fwd_kernel(op, a, b, out) == "transpose", (op, yname, xa, oname)
                    zr.zr_binary_fwd(op, a, b, out=out)
                    bitexact(out.cpu().numpy(), oracle.binary_fwd(op, a.cpu(), b.cpu()),
                             f"transpose {op} y={yname} x_is_a={xa} out={oname}")


def test_planner_occupancy_matches_runtime():
    """The planner sizes grids in whole waves of 152 x (resident CTAs per SM);
    its per-kernel occupancy must be what the runtime reports on this GPU."""
    L = zr.lib()
    L.zr_test_occupancy.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                    ctypes.POINTER(ctypes.c_int)]
    for which in range(28):
        planned, actual = ctypes.c_int(0), ctypes.c_int(0)
        assert L.zr_test_occupancy(which, ctypes.byref(planned), ctypes.byref(actual)) == 0
        assert planned.value == actual.value, (which, planned.value, actual.value)
    assert L.zr_test_occupancy(28, ctypes.byref(planned), ctypes.byref(actual)) == -4


def test_strided_output_and_in_place():
    rng = np.random.default_rng(9)
    a = torch.from_numpy(rng.standard_normal((33, 65)).astype(np.float32)).cuda()
    b = torch.from_numpy(rng.standard_normal((65,)).astype(np.float32)).cuda()
    out_store = torch.empty((65, 33), device="cuda")
    out = out_store.t()
    zr.zr_binary_fwd("sub", a, b, out=out)
    bitexact(out.cpu().numpy(), oracle.binary_fwd("sub", a.cpu(), b.cpu()), "strided out")
    ref = oracle.binary_fwd("mul", a.cpu(), b.cpu())
    zr.zr_binary_fwd("mul", a, b, out=a)  # in place
    bitexact(a.cpu().numpy(), ref, "in place")


def test_misaligned_pointers():
    rng = np.random.default_rng(10)
    base = torch.from_numpy(rng.standard_normal(4096 * 3 + 1).astype(np.float32)).cuda()
    a = base[1:1 + 4096 * 3].view(3, 4096)
    b = torch.from_numpy(rng.standard_normal(4096).astype(np.float32)).cuda()
    bitexact(zr.zr_binary_fwd("div", a, b).cpu().numpy(), oracle.binary_fwd("div", a.cpu(), b.cpu()))
    ga, gb = zr.zr_binary_bwd("mul", a, a, b)
    ra, rb, _, sb = oracle.binary_bwd("mul", a.cpu(), a.cpu(), b.cpu())
    bitexact(ga.cpu().numpy(), ra)
    within(gb.cpu().numpy(), rb, sb)


def test_deterministic_backward():
    host = workloads.make_inputs("c3", B=4, T=513, C=768)
    g, x, gamma = host["g"].cuda(), host["x"].cuda(), host["gamma"].cuda()
    r1 = zr.zr_binary_bwd("mul", g, x, gamma)
    r2 = zr.zr_binary_bwd("mul", g, x, gamma)
    for u, v in zip(r1, r2):
        assert torch.equal(u.view(torch.int32), v.view(torch.int32))


def test_errors_on_device_path():
    x = torch.randn(8, 8).cuda()
    L = zr.lib()
    h = torch.randn(8, 8)  # host memory, not addressable as device memory
    dx, kx = zr._desc(x)
    dh, kh = zr._desc(h, need_data=False)
    dh.data = h.data_ptr()
    out = torch.empty(8, 8, device="cuda")
    assert L.zr_binary_fwd(0, dx, dh, out.data_ptr(), None, None) == -6
    g = torch.randn(64, 256).cuda()
    xx = torch.randn(64, 256).cuda()
    bias = torch.randn(256).cuda()
    dg, _ = zr._desc(g)
    dxx, _ = zr._desc(xx)
    db, _ = zr._desc(bias)
    need = ctypes.c_size_t(0)
    ga = torch.empty_like(xx)
    gb = torch.empty_like(bias)
    assert L.zr_binary_bwd(0, dg, dxx, db, ga.data_ptr(), gb.data_ptr(), None, ctypes.byref(need), None) == 0
    if need.value > 0:
        ws = torch.empty(need.value, dtype=torch.uint8, device="cuda")
        small = ctypes.c_size_t(need.value - 16)
        assert L.zr_binary_bwd(0, dg, dxx, db, ga.data_ptr(), gb.data_ptr(), ws.data_ptr(),
                               ctypes.byref(small), None) == -7


SAB_SHAPES = [
    ((2, 1, 256, 4), (1, 3, 1, 4)),
    ((8, 1, 64, 1, 32), (1, 5, 1, 7, 32)),
    ((1, 1, 4, 1, 8, 1, 32, 64), (1, 3, 1, 4, 1, 5, 1, 64)),
    ((3, 1, 16, 1, 8, 1, 64), (1, 4, 1, 5, 1, 3, 64)),
]


@pytest.mark.parametrize("op", OPS)
def test_both_reduced_fused_pass(op):
    """Shapes where both gradients are reduced and the fused one-pass kernel
    is chosen (many CTAs per tile, split dims), element by element."""
    rng = np.random.default_rng(300 + OPS.index(op))
    for sa, sb in SAB_SHAPES:
        a = torch.from_numpy(rng.standard_normal(sa).astype(np.float32))
        b = torch.from_numpy((np.sign(rng.standard_normal(sb)) * (0.5 + rng.random(sb))).astype(np.float32))
        g = torch.from_numpy(rng.standard_normal(np.broadcast_shapes(sa, sb)).astype(np.float32))
        out = zr.zr_binary_fwd(op, a.cuda(), b.cuda()).cpu().numpy()
        bitexact(out, oracle.binary_fwd(op, a, b), f"split fwd {op} {sa} {sb}")
        ga, gb = zr.zr_binary_bwd(op, g.cuda(), a.cuda(), b.cuda())
        ra, rb, s1, s2 = oracle.binary_bwd(op, g, a, b)
        within(ga.cpu().numpy(), ra, s1, f"fused {op} grad_a {sa} {sb}")
        within(gb.cpu().numpy(), rb, s2, f"fused {op} grad_b {sa} {sb}")
        # Deterministic: a second call gives the same bits.
        ga2, gb2 = zr.zr_binary_bwd(op, g.cuda(), a.cuda(), b.cuda())
        assert torch.equal(ga.view(torch.int32), ga2.view(torch.int32))
        assert torch.equal(gb.view(torch.int32), gb2.view(torch.int32))


def _bwd_plans(op, g, a, b, ga, gb):
    L = zr.lib()
    L.zr_test_describe_bwd.argtypes = [ctypes.c_int, zr.ZrTensor, zr.ZrTensor, zr.ZrTensor,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                       ctypes.c_size_t]
    dg, kg = zr._desc(g)
    da, ka = zr._desc(a)
    db, kb = zr._desc(b)
    buf = ctypes.create_string_buffer(16384)
    assert L.zr_test_describe_bwd(zr.OPS[op], dg, da, db, ga.data_ptr(), gb.data_ptr(), buf,
                                  16384) == 0
    return json.loads(buf.value.decode())["plans"]


def _sum_plan(x, shape):
    L = zr.lib()
    L.zr_test_describe_sum.argtypes = [zr.ZrTensor, ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p,
                                       ctypes.c_char_p, ctypes.c_size_t]
    dx, kx = zr._desc(x)
    out = torch.empty(shape, device="cuda")
    buf = ctypes.create_string_buffer(16384)
    assert L.zr_test_describe_sum(dx, len(shape), zr._i64(shape), out.data_ptr(), buf,
                                  16384) == 0
    return json.loads(buf.value.decode())["plans"][0]


CLUSTER_SHAPES = [
    ((256, 1024), (1024,)),          # inner dim kept, 2 column blocks
    ((2048, 1024), (1024,)),
    ((4096, 1024), (1024,)),         # partial slots (too many tiles for clusters)
    ((16, 1024, 768), (768,)),
    ((3, 97, 772), (772,)),
    ((517, 1028), (1028,)),          # ragged rows and column tiles
    ((1028,), (517, 1028)),          # grad_a reduced
    ((128, 256, 512), (1, 256, 1)),  # inner dim reduced
    ((64, 200, 256), (1, 200, 1)),
    ((8, 100, 1024), (1, 100, 1)),
    ((1, 333, 1), (40, 333, 128)),   # too many tiles for a cluster plan
]


@pytest.mark.parametrize("op", OPS)
def test_cluster_reduction(op):
    """Backward plans whose reduced gradient is summed by thread-block
    clusters (no partial slots, no second pass), element by element against
    the oracle, and bitwise stable across calls."""
    rng = np.random.default_rng(400 + OPS.index(op))
    seen = set()
    for sa, sb in CLUSTER_SHAPES:
        a = torch.from_numpy(rng.standard_normal(sa).astype(np.float32))
        b = torch.from_numpy((np.sign(rng.standard_normal(sb)) * (0.5 + rng.random(sb))).astype(np.float32))
        g = torch.from_numpy(rng.standard_normal(np.broadcast_shapes(sa, sb)).astype(np.float32))
        ga_d, gb_d = torch.empty(sa, device="cuda"), torch.empty(sb, device="cuda")
        ad, bd, gd = a.cuda(), b.cuda(), g.cuda()
        for plan in _bwd_plans(op, gd, ad, bd, ga_d, gb_d):
            if plan.get("cluster", 1) > 1:
                assert plan["nslots"] == 1 and plan["ws_bytes"] == 0, plan
                seen.add(plan["inner_kept"])
        ga, gb = zr.zr_binary_bwd(op, gd, ad, bd, grad_a=ga_d, grad_b=gb_d)
        ra, rb, s1, s2 = oracle.binary_bwd(op, g, a, b)
        for which, got, ref, sabs, shape in ((0, ga, ra, s1, sa), (1, gb, rb, s2, sb)):
            reduced = int(np.prod(shape)) != g.numel()
            what = f"cluster {op} grad_{'ab'[which]} {sa} {sb}"
            if is_single_op_grad(op, which, reduced):
                bitexact(got.cpu().numpy(), ref, what)
            else:
                within(got.cpu().numpy(), ref, sabs, what)
        ga2, gb2 = zr.zr_binary_bwd(op, gd, ad, bd)
        assert torch.equal(ga.view(torch.int32), ga2.view(torch.int32))
        assert torch.equal(gb.view(torch.int32), gb2.view(torch.int32))
    # Cluster plans with the inner dim kept and with it reduced were covered.
    assert seen == {0, 1}, seen


def test_cluster_sum_to_shape():
    rng = np.random.default_rng(17)
    for shape, target in (((2048, 1024), (1024,)), ((517, 1028), (1, 1028)),
                          ((8, 100, 1024), (1, 100, 1)), ((128, 256, 512), (1, 256, 1))):
        x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
        xd = x.cuda()
        plan = _sum_plan(xd, target)
        assert plan.get("cluster", 1) > 1, plan
        got = zr.zr_sum_to_shape(xd, target).cpu().numpy()
        ref, sabs = oracle.sum_to_shape(x, target)
        within(got, ref, sabs, f"cluster sum_to_shape {shape}->{target}")


def _rand_bits(rng, shape):
    return rng.integers(0, 2 ** 32, size=shape, dtype=np.uint64).astype(np.uint32).view(np.float32)


def _log_uniform(rng, shape, lo=-60, hi=60):
    mag = np.exp2(rng.uniform(lo, hi, size=shape)).astype(np.float32)
    return np.where(rng.random(shape) < 0.5, -mag, mag).astype(np.float32)


def test_division_is_ieee_bit_exact():
    """Forward div, and the dense g/b gradient, must equal IEEE division bit
    for bit (any NaN matching any NaN): every binade, subnormals, infinities
    and zeros (random bit patterns), broadcast divisors, and divisors +-2^k
    at the ends of the exponent range (2^-126, 2^127, the subnormal 2^-127)."""
    rng = np.random.default_rng(2024)
    cases = []
    cases.append((_rand_bits(rng, (4096, 256)), _rand_bits(rng, (256,))))         # row divisor
    cases.append((_log_uniform(rng, (4096, 256)), _log_uniform(rng, (256,))))     # fast path
    cases.append((_log_uniform(rng, (2048, 512)), _log_uniform(rng, (2048, 1))))  # column divisor
    cases.append((_rand_bits(rng, (1 << 20,)), _rand_bits(rng, (1 << 20,))))      # no reuse
    cases.append((_log_uniform(rng, (1 << 20,), -126, 127), _log_uniform(rng, (1 << 20,), -126, 127)))
    for s in (8.0, 3.0, 1e-40, 3e38, -7.5, 0.0, float("inf")):
        cases.append((_log_uniform(rng, (1 << 18,), -80, 80), np.array([s], np.float32)))
    for s in (2.0 ** -126, 2.0 ** 127, -(2.0 ** -126), 2.0 ** -127, 0.5, -1.0, 1.0, 2.0 ** 64, 0.125):
        cases.append((_rand_bits(rng, (1 << 18,)), np.array([s], np.float32)))
    pow2_rows = (np.float32(2.0) ** rng.integers(-126, 128, 256).astype(np.float32)) * np.sign(
        rng.standard_normal(256)).astype(np.float32)
    cases.append((_rand_bits(rng, (2048, 256)), pow2_rows.astype(np.float32)))
    for a, b in cases:
        ta, tb = torch.from_numpy(a), torch.from_numpy(b)
        got = zr.zr_binary_fwd("div", ta.cuda(), tb.cuda()).cpu().numpy()
        bitexact(got, oracle.binary_fwd("div", ta, tb), f"div {a.shape} / {b.shape}")
        if b.size > 1 and b.size == a.size:
            continue
        # The dense gradient g / b of the same division (b broadcast: grad_b
        # is a sum, compared elsewhere).
        g = torch.from_numpy(_rand_bits(rng, a.shape))
        ga, _ = zr.zr_binary_bwd("div", g.cuda(), ta.cuda(), tb.cuda(), want_b=False)
        ra, _, _, _ = oracle.binary_bwd("div", g, ta, tb, want_b=False)
        bitexact(ga.cpu().numpy(), ra, f"div grad_a {a.shape} / {b.shape}")


def test_sum_to_shape_batched_matmul_broadcast_grads():
    """A weight broadcast over a batched matmul's batch dims gets the sum of
    the per-batch gradients (Operator page, 广播: SumToSize back to the
    weight's shape).  The per-batch products are given; the reduction is
    zr_sum_to_shape: [B, K, N] -> [K, N], [B, H, K, N] -> [1, H, K, N] and
    [B, H, K, N] -> [K, N]."""
    rng = np.random.default_rng(60)
    for shape, target in (((8, 768, 3072), (768, 3072)), ((4, 12, 64, 1024), (1, 12, 64, 1024)),
                          ((4, 12, 64, 1024), (64, 1024)), ((3, 5, 129, 67), (129, 67))):
        x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32))
        got = zr.zr_sum_to_shape(x.cuda(), target).cpu().numpy()
        ref, sabs = oracle.sum_to_shape(x, target)
        within(got, ref, sabs, f"batch-broadcast grad {shape}->{target}")
