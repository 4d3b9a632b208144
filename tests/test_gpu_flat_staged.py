"""GPU parity of two kernel paths against the CPU oracle, on shapes chosen so
that the planner takes them (checked through the plan description first):

* the flat elementwise kernel (problems that coalesce to at most one outer
  dim): ragged item counts, one-element vectors, a column-broadcast operand,
  a scalar, row-strided and misaligned views, bfloat16 storage;
* reductions whose loads are staged through shared memory: inner dim
  reduced with and without partial slots, inner dim kept, one and two
  streamed inputs, float and bfloat16, and more rows per CTA than one offset
  table holds (the table is refilled in chunks, the staging ring restarted).

Forward outputs and one-operation gradients must be bit-identical to the
oracle; summed gradients within 1e-5 * sum|terms| (plus one bf16 unit in
the last place for bf16 storage).
"""
import ctypes
import json

import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
from parity import bitexact, within

pytestmark = pytest.mark.gpu

OPS = {"add": 0, "sub": 1, "mul": 2, "div": 3}


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    lib = zr.lib()
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.zr_test_describe_fwd.argtypes = [ctypes.c_int, zr.ZrTensor, zr.ZrTensor, ctypes.c_void_p,
                                         i64p, ctypes.c_char_p, ctypes.c_size_t]
    lib.zr_test_describe_bwd_t.argtypes = [ctypes.c_int, ctypes.c_int, zr.ZrTensor, zr.ZrTensor,
                                           zr.ZrTensor, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_char_p, ctypes.c_size_t]
    return lib


def _rand(gen, shape, positive_divisor=False):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if positive_divisor:  # |b| in [0.5, 1.5], random sign
        u = torch.rand(shape, generator=gen, dtype=torch.float32) + 0.5
        s = torch.randint(0, 2, shape, generator=gen).to(torch.float32) * 2 - 1
        x = u * s
    return x


def _to_dev(x, dtype=torch.float32):
    """Device copy keeping strides and storage offset."""
    st = x.untyped_storage()
    flat = torch.empty(0, dtype=x.dtype).set_(st, 0, (st.nbytes() // x.element_size(),), (1,))
    return flat.to(dtype).cuda().as_strided(x.shape, x.stride(), x.storage_offset())


def _bf(x):
    """bf16-representable float32 copy of x (same strides)."""
    st = x.untyped_storage()
    flat = torch.empty(0, dtype=x.dtype).set_(st, 0, (st.nbytes() // 4,), (1,))
    r = torch.from_numpy(oracle.round_bf16(flat.numpy()))
    return r.as_strided(x.shape, x.stride(), x.storage_offset())


def _fwd_plan(L, op, a, b, out):
    da, ka = zr._desc(a)
    db, kb = zr._desc(b)
    buf = ctypes.create_string_buffer(4096)
    rc = L.zr_test_describe_fwd(OPS[op], da, db, out.data_ptr(), None, buf, len(buf))
    assert rc == 0, L.zr_status_string(rc)
    return json.loads(buf.value)


def _bwd_plan(L, op, g, a, b, ga, gb):
    dtype = 1 if g.dtype == torch.bfloat16 else 0
    dg, kg = zr._desc(g)
    da, ka = zr._desc(a)
    db, kb = zr._desc(b)
    buf = ctypes.create_string_buffer(16384)
    rc = L.zr_test_describe_bwd_t(dtype, OPS[op], dg, da, db, ga.data_ptr(), gb.data_ptr(), buf,
                                  len(buf))
    assert rc == 0, L.zr_status_string(rc)
    return json.loads(buf.value)


def _views(gen):
    """(name, a, b) host operands whose forward coalesces to at most one
    outer dim."""
    base = _rand(gen, (333, 1030 + 6))
    misaligned = _rand(gen, (333 * 1030 + 1,))[1:].view(333, 1030)
    return [
        ("bias rows, ragged", _rand(gen, (333, 1030)), _rand(gen, (1030,), True)),
        ("one-element vectors", _rand(gen, (97, 1031)), _rand(gen, (1031,), True)),
        ("column broadcast", _rand(gen, (333, 1028)), _rand(gen, (333, 1), True)),
        ("scalar", _rand(gen, (5, 7, 1111)), torch.tensor([0.75])),
        ("same shape", _rand(gen, (1, 70001)), _rand(gen, (1, 70001), True)),
        ("row-strided view", base[:, 3:1033], _rand(gen, (1030,), True)),
        ("misaligned base", misaligned, _rand(gen, (1030,), True)),
    ]


@pytest.mark.parametrize("op", list(OPS))
def test_flat_forward_layouts(L, op):
    gen = torch.Generator().manual_seed(2024 + OPS[op])
    for name, a, b in _views(gen):
        da, db = _to_dev(a), _to_dev(b)
        shape = tuple(np.broadcast_shapes(tuple(a.shape), tuple(b.shape)))
        out = torch.empty(shape, device="cuda")
        plan = _fwd_plan(L, op, da, db, out)
        assert plan["kernel"] == "flat", (name, plan)
        got = zr.zr_binary_fwd(op, da, db, out=out)
        torch.cuda.synchronize()
        bitexact(got.cpu().numpy(), oracle.binary_fwd(op, a, b), f"flat {op} {name}")


@pytest.mark.parametrize("op", list(OPS))
def test_flat_forward_bf16(L, op):
    gen = torch.Generator().manual_seed(3030 + OPS[op])
    for name, a, b in _views(gen):
        a16, b16 = _bf(a), _bf(b)
        da, db = _to_dev(a16, torch.bfloat16), _to_dev(b16, torch.bfloat16)
        got = zr.zr_binary_fwd(op, da, db)
        torch.cuda.synchronize()
        ref = oracle.round_bf16(oracle.binary_fwd(op, a16, b16))
        bitexact(got.float().cpu().numpy(), ref, f"flat bf16 {op} {name}")


# (g shape, b shape), a has g's shape.  Staged in bf16 for every op and in
# float for add; in float the two narrow inner-kept cases of mul and div run
# three CTAs per SM and stay under two waves, so they load into registers.
STAGED = [
    ((3, 700, 4096), (1, 700, 1)),      # inner dim reduced, 3 partial slots
    ((1300, 2048), (1300, 1)),          # inner dim reduced, one CTA per output
    ((64, 16400, 8), (64, 1, 8)),       # inner dim kept, 864 rows per CTA: two table chunks
    ((1024, 1100, 8), (1024, 1, 8)),    # inner dim kept, 550 rows per CTA, 2 slots
]


def _staged_case(L, op, gshape, bshape, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    g = _rand(gen, gshape)
    a = _rand(gen, gshape)
    b = _rand(gen, bshape, positive_divisor=True)
    if dtype == torch.bfloat16:
        g, a, b = _bf(g), _bf(a), _bf(b)
    dg, da, db = _to_dev(g, dtype), _to_dev(a, dtype), _to_dev(b, dtype)
    ga = torch.empty(gshape, dtype=dtype, device="cuda")
    gb = torch.empty(bshape, dtype=dtype, device="cuda")
    plan = _bwd_plan(L, op, dg, da, db, ga, gb)
    staged = [p for p in plan["plans"] if p.get("stages", 0) >= 2]
    got_a, got_b = zr.zr_binary_bwd(op, dg, da, db, grad_a=ga, grad_b=gb)
    torch.cuda.synchronize()
    ra, rb, sa, sb = oracle.binary_bwd(op, g, a, b)
    bf = dtype == torch.bfloat16
    if bf:
        ra, rb = oracle.round_bf16(ra), oracle.round_bf16(rb)
    what = f"staged {op} {gshape}->{bshape} {'bf16' if bf else 'f32'}"
    # grad_a is dense: one operation per element (g, g*b or g/b)
    bitexact(got_a.float().cpu().numpy(), ra, what + " grad_a")
    extra = (2.0 ** -7 / 1e-5) * np.abs(np.asarray(rb, np.float64)) if bf else 0.0
    within(got_b.float().cpu().numpy(), rb, sb + extra, what + " grad_b")
    return staged


@pytest.mark.parametrize("op", ["add", "mul", "div"])
def test_staged_reductions_f32(L, op):
    n_staged = 0
    for i, (gs, bs) in enumerate(STAGED):
        staged = _staged_case(L, op, gs, bs, torch.float32, 4040 + 10 * i + OPS[op])
        n_staged += bool(staged)
        if op == "add" and gs == (64, 16400, 8):
            # Staged, with the offset table refilled: 864 rows per CTA.
            assert staged and staged[0]["rows_per_blk"] > 512 and staged[0]["nslots"] > 1, staged
    # Inner-reduced plans (with and without slots) are staged for every op.
    assert n_staged >= 2


@pytest.mark.parametrize("op", ["add", "mul", "div"])
def test_staged_reductions_bf16(L, op):
    for i, (gs, bs) in enumerate(STAGED):
        staged = _staged_case(L, op, gs, bs, torch.bfloat16, 5050 + 10 * i + OPS[op])
        assert staged, (op, gs, bs)


def _special_dividends(gen, n):
    x = torch.randn(n, generator=gen, dtype=torch.float32)
    specials = torch.tensor([0.0, -0.0, float("inf"), -float("inf"), float("nan"), 1e-40, -3e-42,
                             1.2e-38, -1.1754944e-38, 3.0e38, -3.4e38, 1.0, -2.5, 6e-39, 2.0 ** -149],
                            dtype=torch.float32)
    x[: specials.numel()] = specials
    x[-specials.numel():] = specials
    return x


# One-element divisors: powers of two whose reciprocal is normal take one
# multiplication by the exact reciprocal; the rest (2^127, a subnormal,
# zeros, infinities, NaN, non-powers of two) the IEEE division.
DIVISORS = [8.0, -0.25, 2.0 ** -126, 2.0 ** 126, 1.0, -1.0, 2.0 ** 127, 2.0 ** -127, 3.0, -0.0,
            float("inf"), float("nan"), 0.1]


@pytest.mark.parametrize("bf16", [False, True])
def test_division_by_one_element_divisors_forward(L, bf16):
    gen = torch.Generator().manual_seed(6060)
    for shape in [(7, 1031), (96, 4096)]:  # a ragged tail; 16-byte vectors
        a = _special_dividends(gen, int(np.prod(shape))).view(shape)
        if bf16:
            a = _bf(a)
        for d in DIVISORS:
            b = torch.tensor([d], dtype=torch.float32)
            if bf16:
                b = _bf(b)
            dt = torch.bfloat16 if bf16 else torch.float32
            got = zr.zr_binary_fwd("div", _to_dev(a, dt), _to_dev(b, dt))
            torch.cuda.synchronize()
            ref = oracle.binary_fwd("div", a, b)
            if bf16:
                ref = oracle.round_bf16(ref)
            bitexact(got.float().cpu().numpy(), ref, f"x / {d!r} {shape} {'bf16' if bf16 else 'f32'}")


@pytest.mark.parametrize("bf16", [False, True])
def test_division_by_one_element_divisors_backward(L, bf16):
    """grad_a = g / b is dense (bit-exact); grad_b = -sum(g * a) / b^2 is summed."""
    gen = torch.Generator().manual_seed(7070)
    dt = torch.bfloat16 if bf16 else torch.float32
    for shape in [(7, 1031), (3, 700, 4096)]:  # register loads; a staged grid
        n = int(np.prod(shape))
        # Moderate values with signed zeros and subnormals (huge ones would
        # overflow the binary32 sums that the binary64 oracle keeps finite).
        g = torch.randn(n, generator=gen, dtype=torch.float32)
        g[:6] = torch.tensor([0.0, -0.0, 1e-40, -3e-42, 1.2e-38, 2.0 ** -149])
        g = g.view(shape)
        a = torch.randn(shape, generator=gen, dtype=torch.float32)
        if bf16:
            g, a = _bf(g), _bf(a)
        for d in [8.0, -0.25, 2.0 ** -60, 2.0 ** 60, 3.0, 2.0 ** 127]:
            b = torch.tensor([d], dtype=torch.float32)
            if bf16:
                b = _bf(b)
            ga, gb = zr.zr_binary_bwd("div", _to_dev(g, dt), _to_dev(a, dt), _to_dev(b, dt))
            torch.cuda.synchronize()
            ra, rb, sa, sb = oracle.binary_bwd("div", g, a, b)
            what = f"g / {d!r} {shape} {'bf16' if bf16 else 'f32'}"
            if bf16:
                ra, rb = oracle.round_bf16(ra), oracle.round_bf16(rb)
            bitexact(ga.float().cpu().numpy(), ra, what + " grad_a")
            extra = (2.0 ** -7 / 1e-5) * np.abs(np.asarray(rb, np.float64)) if bf16 else 0.0
            within(gb.float().cpu().numpy(), rb, sb + extra, what + " grad_b")


def _halves(shape, axis, big=1000.0):
    """+big in the first half along `axis`, -big in the second: every sum
    over that axis cancels exactly to 0 while each half alone is large."""
    g = torch.full(shape, big, dtype=torch.float32)
    idx = [slice(None)] * len(shape)
    idx[axis] = slice(shape[axis] // 2, None)
    g[tuple(idx)] = -big
    return g


def _chain_plan(L, op1, op2, g, a, b, c, grads):
    L.zr_test_describe_chain_bwd.argtypes = [ctypes.c_int, ctypes.c_int, zr.ZrTensor, zr.ZrTensor,
                                             zr.ZrTensor, zr.ZrTensor, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                             ctypes.c_size_t]
    keep = [zr._desc(x) for x in (g, a, b, c)]
    buf = ctypes.create_string_buffer(8192)
    rc = L.zr_test_describe_chain_bwd(OPS[op1], OPS[op2], *[k[0] for k in keep],
                                      *[x.data_ptr() for x in grads], buf, len(buf))
    assert rc == 0, L.zr_status_string(rc)
    return json.loads(buf.value)


def test_division_factor_applies_to_each_total(L):
    """Division's summed gradient is -sum(g * a) / b^2: the factor 1/b^2
    multiplies the whole sum once.  With b = 2^-60 and sums whose halves are
    large and cancel exactly, the factor times any partial sum overflows
    binary32 while the true gradient is 0; every route with partial sums
    must still give 0 (the oracle's binary64 value), not inf - inf = NaN."""
    tiny = 2.0 ** -60
    # Reductions with partial slots: inner dim kept, and reduced.
    for gshape, bshape, axis in [((4096, 1024), (1024,), 0), ((3, 700, 4096), (1, 700, 1), 0)]:
        g = _halves(gshape, axis)
        if gshape[0] == 3:
            g[2] = 0.0
        a = torch.ones(gshape)
        b = torch.full(bshape, tiny)
        dg, da, db = _to_dev(g), _to_dev(a), _to_dev(b)
        ga = torch.empty(gshape, device="cuda")
        gb = torch.empty(bshape, device="cuda")
        plan = _bwd_plan(L, "div", dg, da, db, ga, gb)
        assert plan["plans"][0]["nslots"] > 1, plan
        zr.zr_binary_bwd("div", dg, da, db, grad_a=ga, grad_b=gb)
        torch.cuda.synchronize()
        ra, rb, sa, sb = oracle.binary_bwd("div", g, a, b)
        bitexact(ga.cpu().numpy(), ra, f"div {gshape} grad_a")
        within(gb.cpu().numpy(), rb, sb, f"div {gshape} grad_b")
        assert np.all(rb == 0.0) and np.all(gb.cpu().numpy() == 0.0)
    # Both gradients reduced (the two-gradient pass): grad_b's slots are
    # a's outer tiles, so halves along a's outermost dim cancel.
    sa_, sb_ = (2, 1, 4, 1, 8, 1, 16, 32), (1, 3, 1, 5, 1, 6, 1, 32)
    gshape = tuple(np.broadcast_shapes(sa_, sb_))
    g, a, b = _halves(gshape, 0), torch.ones(sa_), torch.full(sb_, tiny)
    dg, da, db = _to_dev(g), _to_dev(a), _to_dev(b)
    ga, gb = torch.empty(sa_, device="cuda"), torch.empty(sb_, device="cuda")
    assert _bwd_plan(L, "div", dg, da, db, ga, gb)["plans"][0]["kernel"] == "sab"
    zr.zr_binary_bwd("div", dg, da, db, grad_a=ga, grad_b=gb)
    torch.cuda.synchronize()
    ra, rb, sa, sb = oracle.binary_bwd("div", g, a, b)
    within(ga.cpu().numpy(), ra, sa, "sab div grad_a")
    within(gb.cpu().numpy(), rb, sb, "sab div grad_b")
    assert np.all(rb == 0.0) and np.all(gb.cpu().numpy() == 0.0)
    # Fused chains: (a + b) / c with c one element (per-CTA partials), and
    # (a * b) / c with c shaped like b (slot rows of grad_b and grad_c).
    R, C = 4096, 1024
    for op1, cshape in [("add", (1,)), ("mul", (C,))]:
        g = _halves((R, C), 0)
        a = torch.ones((R, C))
        b = torch.zeros((C,)) if op1 == "add" else torch.ones((C,))
        c = torch.full(cshape, tiny)
        dg, da, db, dc = _to_dev(g), _to_dev(a), _to_dev(b), _to_dev(c)
        grads = [torch.empty((R, C), device="cuda"), torch.empty((C,), device="cuda"),
                 torch.empty(cshape, device="cuda")]
        plan = _chain_plan(L, op1, "div", dg, da, db, dc, grads)
        assert plan["route"] == "fused", plan
        zr.zr_chain_bwd(op1, "div", dg, da, db, dc, grads=tuple(grads))
        torch.cuda.synchronize()
        refs = oracle.chain_bwd(op1, "div", g, a, b, c)
        what = f"chain ({op1}, div) c {cshape}"
        bitexact(grads[0].cpu().numpy(), refs[0], what + " grad_a")
        for k in (1, 2):
            within(grads[k].cpu().numpy(), refs[k], refs[k + 3], what + f" grad_{'abc'[k]}")
            assert np.all(grads[k].cpu().numpy() == 0.0), what
