"""Host-side checks of the C ABI library (no GPU needed).

* the library loads and exports every function declared in include/*.h;
* zr_broadcast_shape agrees with the book's printed examples and NumPy;
* the multiply-high division used by the kernels is exact;
* a host walk of every planned kernel (the same CTA/item/row/column loops the
  kernels run, via zr_test_emulate_*) visits each output element exactly
  once and computes the same operand offsets and gradient indices as naive
  strided index arithmetic written here with NumPy;
* argument errors are reported before anything touches a device.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import broadcast_elementwise_shape_gb300 as zr
from broadcast_elementwise_shape_gb300 import ZrTensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    zr.build()
    lib = zr.lib()
    i64p = ctypes.POINTER(ctypes.c_int64)
    vp = ctypes.c_void_p
    lib.zr_test_fastdiv.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]
    lib.zr_test_describe_fwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, vp, i64p, ctypes.c_char_p, ctypes.c_size_t]
    lib.zr_test_describe_bwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, ZrTensor, vp, vp, ctypes.c_char_p, ctypes.c_size_t]
    lib.zr_test_describe_sum.argtypes = [ZrTensor, ctypes.c_int32, i64p, vp, ctypes.c_char_p, ctypes.c_size_t]
    lib.zr_test_emulate_fwd.argtypes = [ZrTensor, ZrTensor, vp, i64p, ctypes.c_int64, i64p, i64p]
    lib.zr_test_emulate_bwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, ZrTensor, vp, vp, ctypes.c_int64, i64p, i64p]
    return lib


def _i64(seq):
    return (ctypes.c_int64 * max(1, len(seq)))(*[int(v) for v in seq])


class FakeT:
    """A descriptor with a fake (never dereferenced) base address."""

    def __init__(self, addr, shape, strides=None):
        self.shape = tuple(shape)
        self.strides = tuple(strides) if strides is not None else tuple(
            s // 4 for s in np.empty(self.shape, np.float32).strides) if self.shape else ()
        self._sz = _i64(self.shape)
        self._st = _i64(self.strides)
        self.desc = ZrTensor(addr, len(self.shape), self._sz, self._st)


def declared_functions():
    names = []
    for f in os.listdir(INCLUDE):
        if f.endswith(".h"):
            text = open(os.path.join(INCLUDE, f)).read()
            names += re.findall(r"^\s*(?:int|const char\*)\s+(zr_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"zr_broadcast_shape", "zr_binary_fwd", "zr_binary_bwd", "zr_sum_to_shape",
            "zr_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(0, -10, -1):
        assert L.zr_status_string(code).decode().startswith("ZR_")


def test_broadcast_shape_examples_and_numpy(L):
    assert zr.zr_broadcast_shape((2, 3, 4), (3, 1)) == (2, 3, 4)
    with pytest.raises(zr.ZrError) as e:
        zr.zr_broadcast_shape((2, 3, 4), (2, 4, 5))
    assert e.value.status == -3
    rng = np.random.default_rng(0)
    for _ in range(2000):
        na, nb = rng.integers(0, 9, 2)
        sa = tuple(int(v) for v in rng.choice([0, 1, 1, 2, 3, 5], na))
        sb = tuple(int(v) for v in rng.choice([0, 1, 1, 2, 3, 5], nb))
        try:
            ref = tuple(np.broadcast_shapes(sa, sb))
        except ValueError:
            ref = None
        if ref is None:
            with pytest.raises(zr.ZrError):
                zr.zr_broadcast_shape(sa, sb)
        else:
            assert zr.zr_broadcast_shape(sa, sb) == ref
    with pytest.raises(zr.ZrError) as e:
        zr.zr_broadcast_shape((1,) * 9, (1,))
    assert e.value.status == -2


def test_fastdiv_exact(L):
    rng = np.random.default_rng(1)
    q = ctypes.c_uint32()
    ds = [1, 2, 3, 5, 7, 10, 12, 64, 96, 255, 256, 641, 65535, 65536, 2**31 - 1, 2**31,
          2**31 + 1, 2**32 - 1] + [int(v) for v in rng.integers(1, 2**32, 300)]
    ns = [0, 1, 2, 2**31 - 1, 2**31, 2**32 - 2, 2**32 - 1]
    for d in ds:
        for n in ns + [int(v) for v in rng.integers(0, 2**32, 40)] + [d - 1, d, d + 1, 2 * d - 1]:
            if not 0 <= n < 2**32:
                continue
            assert L.zr_test_fastdiv(d, n, ctypes.byref(q)) == 0
            assert q.value == n // d, (d, n)


# ------------------------------------------------------------- naive index maps

def naive_offsets(out_shape, x_shape, x_strides):
    """Element offset of x for every output coordinate (row-major), with
    coordinate 0 on x's size-1 or missing dims."""
    n = len(out_shape)
    off = np.zeros(out_shape, np.int64)
    for od in range(n):
        d = od - (n - len(x_shape))
        if d < 0 or x_shape[d] == 1:
            continue
        shape = [1] * n
        shape[od] = out_shape[od]
        off = off + np.arange(out_shape[od], dtype=np.int64).reshape(shape) * x_strides[d]
    return off


def dense_strides(shape):
    return tuple(s // 4 for s in np.empty(shape, np.float32).strides) if shape else ()


def rand_view(rng, shape, addr):
    """Fake view of `shape`: contiguous, permuted or stepped strides; some
    base addresses are misaligned by one element."""
    kind = rng.integers(0, 3)
    if kind == 0 or len(shape) == 0:
        st = dense_strides(shape)
    elif kind == 1:
        perm = rng.permutation(len(shape))
        base = dense_strides(tuple(shape[p] for p in perm))
        st = [0] * len(shape)
        for i, p in enumerate(perm):
            st[p] = base[i]
        st = tuple(st)
    else:
        big = tuple(2 * s + 1 for s in shape)
        st = tuple(2 * s for s in dense_strides(big))
    return FakeT(addr, shape, st)


def rand_shapes(rng, max_nd=6):
    n = int(rng.integers(0, max_nd + 1))
    out = [int(v) for v in rng.choice([1, 2, 3, 4, 5, 8, 12], n)]
    sa = [s if rng.random() < 0.6 else 1 for s in out]
    sb = [s if rng.random() < 0.6 else 1 for s in out]
    sa = sa[int(rng.integers(0, n + 1)) if n else 0:]
    sb = sb[int(rng.integers(0, n + 1)) if n else 0:]
    return tuple(sa), tuple(sb)


def test_emulated_forward_matches_naive(L):
    rng = np.random.default_rng(2)
    checked = 0
    for it in range(400):
        sa, sb = rand_shapes(rng)
        out_shape = np.broadcast_shapes(sa, sb)
        n_out = int(np.prod(out_shape))
        if n_out == 0:
            continue
        a = rand_view(rng, sa, 0x100000 + 4 * int(rng.integers(0, 2)))
        b = rand_view(rng, sb, 0x900000)
        if rng.random() < 0.5:
            ost = dense_strides(out_shape)
        else:
            ost = rand_view(rng, out_shape, 0).strides
        outp = 0x4000000 + (4 if rng.random() < 0.2 else 0)
        cap = n_out + 8
        rec = (ctypes.c_int64 * (3 * cap))()
        nrec = ctypes.c_int64()
        rc = L.zr_test_emulate_fwd(a.desc, b.desc, outp, _i64(ost), cap, rec, ctypes.byref(nrec))
        assert rc == 0, (sa, sb, rc)
        r = np.frombuffer(rec, np.int64)[: 3 * nrec.value].reshape(-1, 3)
        assert r.shape[0] == n_out
        o = naive_offsets(out_shape, out_shape, ost).ravel()
        ao = naive_offsets(out_shape, sa, a.strides).ravel()
        bo = naive_offsets(out_shape, sb, b.strides).ravel()
        order = np.argsort(r[:, 0])
        ref_order = np.argsort(o)
        np.testing.assert_array_equal(r[order, 0], o[ref_order])
        np.testing.assert_array_equal(r[order, 1], ao[ref_order])
        np.testing.assert_array_equal(r[order, 2], bo[ref_order])
        checked += 1
    assert checked > 250


def grad_index(out_shape, x_shape):
    """Index into x's dense row-major layout for every output coordinate."""
    return naive_offsets(out_shape, x_shape, dense_strides(x_shape))


@pytest.mark.parametrize("op", [0, 1, 2, 3])
def test_emulated_backward_matches_naive(L, op):
    rng = np.random.default_rng(10 + op)
    checked = 0
    for it in range(250):
        sa, sb = rand_shapes(rng)
        out_shape = np.broadcast_shapes(sa, sb)
        n_out = int(np.prod(out_shape))
        if n_out == 0:
            continue
        g = rand_view(rng, out_shape, 0x100000 + 4 * int(rng.integers(0, 2)))
        a = rand_view(rng, sa, 0x2000000)
        b = rand_view(rng, sb, 0x3000000)
        want = int(rng.integers(1, 4))
        pa = 0x5000000 if want & 1 else None
        pb = 0x6000000 if want & 2 else None
        buf = ctypes.create_string_buffer(8192)
        assert L.zr_test_describe_bwd(op, g.desc, a.desc, b.desc, pa, pb, buf, 8192) == 0
        desc = json.loads(buf.value.decode())
        cap = 2 * n_out + 8
        rec = (ctypes.c_int64 * (7 * cap))()
        nrec = ctypes.c_int64()
        rc = L.zr_test_emulate_bwd(op, g.desc, a.desc, b.desc, pa, pb, cap, rec, ctypes.byref(nrec))
        assert rc == 0
        r = np.frombuffer(rec, np.int64)[: 7 * nrec.value].reshape(-1, 7)
        go = naive_offsets(out_shape, out_shape, g.strides).ravel()
        ao = naive_offsets(out_shape, sa, a.strides).ravel()
        bo = naive_offsets(out_shape, sb, b.strides).ravel()
        xa = grad_index(out_shape, sa).ravel()
        xb = grad_index(out_shape, sb).ravel()
        dense = np.arange(n_out, dtype=np.int64)
        ref_by_g = np.argsort(go)
        plans = desc["plans"]
        for pi, plan in enumerate(plans):
            rp = r[r[:, 0] == pi]
            assert rp.shape[0] == n_out, (sa, sb, plan)
            order = np.argsort(rp[:, 1])
            np.testing.assert_array_equal(rp[order, 1], go[ref_by_g])
            rows = rp[order]
            ref = ref_by_g
            if rows[0, 2] != -1:
                np.testing.assert_array_equal(rows[:, 2], ao[ref])
            if rows[0, 3] != -1:
                np.testing.assert_array_equal(rows[:, 3], bo[ref])
            if plan["kernel"] in ("reduce", "sab"):
                which = desc["which"][pi]
                np.testing.assert_array_equal(rows[:, 4], (xa if which == 0 else xb)[ref])
                # slot: the partial the term goes to (a workspace slot, or
                # the CTA's rank in a cluster plan)
                bound = plan["nslots"] if plan.get("cluster", 1) <= 1 else plan["cluster"]
                assert rows[:, 5].min() >= 0 and rows[:, 5].max() < bound
                if plan.get("dense_out"):
                    np.testing.assert_array_equal(rows[:, 6], dense[ref])
            else:
                np.testing.assert_array_equal(rows[:, 6], dense[ref])
        checked += 1
    assert checked > 150


def test_plan_dispatch_for_workloads(L):
    """The five workloads coalesce the way the design expects."""
    T = 1 << 40  # fake base addresses far apart

    def fwd(sa, sb, sta=None):
        a, b = FakeT(T, sa, sta), FakeT(2 * T, sb)
        buf = ctypes.create_string_buffer(4096)
        assert L.zr_test_describe_fwd(2, a.desc, b.desc, 3 * T, None, buf, 4096) == 0
        return json.loads(buf.value.decode())

    def bwd(op, sa, sb, sta=None):
        out = np.broadcast_shapes(sa, sb)
        g, a, b = FakeT(T, out), FakeT(2 * T, sa, sta), FakeT(3 * T, sb)
        buf = ctypes.create_string_buffer(4096)
        assert L.zr_test_describe_bwd(op, g.desc, a.desc, b.desc, 4 * T, 5 * T, buf, 4096) == 0
        return json.loads(buf.value.decode())

    d = fwd((4096, 1024), (1024,))
    assert (d["nrow"], d["ncol"], d["vec"], d["inner_stride"][1]) == (4096, 1024, 4, 1)
    d = fwd((8, 12, 1024, 1024), (1,))
    assert (d["nrow"], d["ncol"], d["inner_stride"][1]) == (1, 8 * 12 * 1024 * 1024, 0)
    d = fwd((8, 12, 1024, 1024), (1, 1, 1024, 1024))
    assert (d["nrow"], d["ncol"]) == (96, 1024 * 1024)
    d = fwd((128, 256, 512), (1, 256, 1), sta=(131072, 1, 256))
    assert d["kernel"] == "transpose" and d["xs_q"] == 256 and (d["np"], d["nq"]) == (256, 512)
    d = fwd((4, 1, 8, 1, 16, 1, 32, 64), (1, 6, 1, 12, 1, 10, 1, 64))
    assert d["kernel"] == "sab_fwd" and (d["ta"], d["n_tiles"], d["n_beta"]) == (128, 128, 720)
    d = bwd(0, (4096, 1024), (1024,))
    (p,) = d["plans"]
    assert p["kernel"] == "reduce" and p["inner_kept"] == 1 and p["dense_out"] == 1
    assert (p["n_kept"], p["n_red"], p["ncol"]) == (1, 4096, 1024)
    d = bwd(1, (128, 256, 512), (1, 256, 1), sta=(131072, 1, 256))
    (p,) = d["plans"]
    assert p["inner_kept"] == 0 and (p["n_kept"], p["n_red"], p["ncol"]) == (256, 128, 512)
    d = bwd(3, (100663296,), (1,))
    (p,) = d["plans"]
    assert p["inner_kept"] == 0 and p["n_kept"] == 1 and p["nout"] == 1


def test_errors_before_any_device_access(L):
    a = FakeT(0x100000, (2, 3, 4))
    b = FakeT(0x200000, (2, 4, 5))
    out = 0x300000
    assert L.zr_binary_fwd(0, a.desc, b.desc, out, None, None) == -3
    bad = ZrTensor(0x100000, 9, _i64([1] * 9), None)
    assert L.zr_binary_fwd(0, bad, b.desc, out, None, None) == -2
    neg = FakeT(0x100000, (2, -1), (1, 1))
    assert L.zr_binary_fwd(0, neg.desc, b.desc, out, None, None) == -4
    assert L.zr_binary_fwd(7, a.desc, a.desc, out, None, None) == -1
    # Output overlapping an input partially.
    x = FakeT(0x100000, (4, 4))
    assert L.zr_binary_fwd(0, x.desc, x.desc, 0x100000 + 4, None, None) == -5
    # Output with a zero stride overlaps itself.
    assert L.zr_binary_fwd(0, x.desc, x.desc, 0x900000, _i64([0, 1]), None) == -5
    # Workspace query is host-only and sizes the partials.
    T = 1 << 40
    g = FakeT(T, (4096, 1024))
    xx = FakeT(2 * T, (4096, 1024))
    bias = FakeT(3 * T, (1024,))
    nbytes = ctypes.c_size_t(0)
    assert L.zr_binary_bwd(0, g.desc, xx.desc, bias.desc, 4 * T, 5 * T, None,
                           ctypes.byref(nbytes), None) == 0
    assert nbytes.value > 0
    # grad_out of the wrong shape.
    g2 = FakeT(T, (4096, 1023))
    assert L.zr_binary_bwd(0, g2.desc, xx.desc, bias.desc, 4 * T, 5 * T, None,
                           ctypes.byref(nbytes), None) == -3
    # Gradients overlapping each other.
    assert L.zr_binary_bwd(0, g.desc, xx.desc, bias.desc, 4 * T, 4 * T + 64, None,
                           ctypes.byref(nbytes), None) == -5
    # sum_to_shape onto a shape that does not broadcast back.
    assert L.zr_sum_to_shape(xx.desc, 1, _i64([1023]), 6 * T, None, ctypes.byref(nbytes), None) == -3


def _dry_lib(L):
    vp = ctypes.c_void_p
    i64p = ctypes.POINTER(ctypes.c_int64)
    L.zr_test_dry_run_fwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, vp, i64p]
    L.zr_test_dry_run_bwd.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, ZrTensor, vp, vp]
    L.zr_test_dry_run_sum.argtypes = [ZrTensor, ctypes.c_int32, i64p, vp]
    return L


NEEDS_A = {0: (False, False), 1: (False, False), 2: (False, True), 3: (False, True)}
NEEDS_B = {0: (False, False), 1: (False, False), 2: (True, False), 3: (True, True)}


@pytest.mark.parametrize("op", [0, 1, 2, 3])
def test_every_plan_provides_what_its_kernels_read(L, op):
    """Plans built with a/b data NULL whenever no requested gradient needs
    them must pass the launch-time operand checks (a kernel that would read a
    missing operand is refused before launch)."""
    L = _dry_lib(L)
    T = 1 << 40
    rng = np.random.default_rng(50 + op)
    shapes = [((4, 1, 8, 1, 16, 1, 32, 64), (1, 6, 1, 12, 1, 10, 1, 64)),
              ((4096, 1024), (1024,)), ((16, 1024, 768), (768,)), ((32, 64, 128), (64, 1)),
              ((8, 12, 1024, 1024), (1, 1, 1024, 1024)), ((100663296,), (1,))]
    for _ in range(150):
        shapes.append(rand_shapes(rng))
    for sa, sb in shapes:
        out_shape = tuple(np.broadcast_shapes(sa, sb))
        if int(np.prod(out_shape)) == 0:
            continue
        for want in (1, 2, 3):
            need_a = (want & 1 and NEEDS_A[op][0]) or (want & 2 and NEEDS_A[op][1])
            need_b = (want & 1 and NEEDS_B[op][0]) or (want & 2 and NEEDS_B[op][1])
            g = FakeT(T, out_shape)
            a = FakeT(2 * T if need_a else None, sa)
            b = FakeT(3 * T if need_b else None, sb)
            pa = 4 * T if want & 1 else None
            pb = 5 * T if want & 2 else None
            assert L.zr_test_dry_run_bwd(op, g.desc, a.desc, b.desc, pa, pb) == 0, (op, want, sa, sb)
        a, b = FakeT(2 * T, sa), FakeT(3 * T, sb)
        assert L.zr_test_dry_run_fwd(op, a.desc, b.desc, 4 * T, None) == 0
        assert L.zr_test_dry_run_sum(g.desc, len(sb), _i64(sb), 6 * T) in (0, -3)


SAB_CASES = [
    ((2, 1, 256, 4), (1, 3, 1, 4)),            # one tile, three steps
    ((8, 1, 64, 1, 32), (1, 5, 1, 7, 32)),     # split A dim, 2 tiles, many CTAs per tile
    ((3, 1, 16, 1, 8, 1, 64), (1, 4, 1, 5, 1, 3, 64)),
]


def test_emulated_split_forward(L):
    """Forward shapes whose outer dims each vary in one input take the split
    kernel; its host walk must write every output once from the right a and b."""
    T = 1 << 40
    for sa, sb in SAB_CASES + [((2, 1, 4, 1, 8, 1, 32, 64), (1, 3, 1, 4, 1, 5, 1, 64))]:
        out_shape = tuple(np.broadcast_shapes(sa, sb))
        n_out = int(np.prod(out_shape))
        a, b = FakeT(T, sa), FakeT(2 * T, sb)
        buf = ctypes.create_string_buffer(4096)
        assert L.zr_test_describe_fwd(3, a.desc, b.desc, 3 * T, None, buf, 4096) == 0
        assert json.loads(buf.value.decode())["kernel"] == "sab_fwd"
        cap = n_out + 8
        rec = (ctypes.c_int64 * (3 * cap))()
        nrec = ctypes.c_int64()
        assert L.zr_test_emulate_fwd(a.desc, b.desc, 3 * T, None, cap, rec, ctypes.byref(nrec)) == 0
        r = np.frombuffer(rec, np.int64)[: 3 * nrec.value].reshape(-1, 3)
        assert r.shape[0] == n_out
        o = naive_offsets(out_shape, out_shape, dense_strides(out_shape)).ravel()
        ao = naive_offsets(out_shape, sa, a.strides).ravel()
        bo = naive_offsets(out_shape, sb, b.strides).ravel()
        order, ref = np.argsort(r[:, 0]), np.argsort(o)
        np.testing.assert_array_equal(r[order, 0], o[ref])
        np.testing.assert_array_equal(r[order, 1], ao[ref])
        np.testing.assert_array_equal(r[order, 2], bo[ref])


@pytest.mark.parametrize("op", [0, 1, 2, 3])
def test_emulated_sab_backward(L, op):
    """Shapes where both gradients are reduced take the fused pass; its host
    walk must visit every grad_out element once with naive offsets and
    gradient indices, and fill every grad_a partial slot exactly once."""
    T = 1 << 40
    for sa, sb in SAB_CASES:
        out_shape = tuple(np.broadcast_shapes(sa, sb))
        n_out = int(np.prod(out_shape))
        g, a, b = FakeT(T, out_shape), FakeT(2 * T, sa), FakeT(3 * T, sb)
        buf = ctypes.create_string_buffer(8192)
        assert L.zr_test_describe_bwd(op, g.desc, a.desc, b.desc, 4 * T, 5 * T, buf, 8192) == 0
        desc = json.loads(buf.value.decode())
        assert [p["kernel"] for p in desc["plans"]] == ["sab", "sab"], desc
        cap = 2 * n_out + 8
        rec = (ctypes.c_int64 * (7 * cap))()
        nrec = ctypes.c_int64()
        assert L.zr_test_emulate_bwd(op, g.desc, a.desc, b.desc, 4 * T, 5 * T, cap, rec,
                                     ctypes.byref(nrec)) == 0
        r = np.frombuffer(rec, np.int64)[: 7 * nrec.value].reshape(-1, 7)
        go = naive_offsets(out_shape, out_shape, g.strides).ravel()
        ao = naive_offsets(out_shape, sa, a.strides).ravel()
        bo = naive_offsets(out_shape, sb, b.strides).ravel()
        xs = (grad_index(out_shape, sa).ravel(), grad_index(out_shape, sb).ravel())
        ref = np.argsort(go)
        for pi in (0, 1):
            rows = r[r[:, 0] == pi]
            assert rows.shape[0] == n_out
            rows = rows[np.argsort(rows[:, 1])]
            np.testing.assert_array_equal(rows[:, 1], go[ref])
            np.testing.assert_array_equal(rows[:, 4], xs[pi][ref])
            if op >= 2:
                np.testing.assert_array_equal(rows[:, 2], ao[ref])
                np.testing.assert_array_equal(rows[:, 3], bo[ref])
            assert rows[:, 5].min() >= 0 and rows[:, 5].max() < desc["plans"][pi]["nslots"]
        L2 = _dry_lib(L)
        need_ab = op >= 2
        a2 = FakeT(2 * T if need_ab else None, sa)
        b2 = FakeT(3 * T if need_ab else None, sb)
        assert L2.zr_test_dry_run_bwd(op, g.desc, a2.desc, b2.desc, 4 * T, 5 * T) == 0


# ---------------------------------------------------------------- two-op chains

def _chain_desc(L, op1, op2, sa, sb, sc, sta=None, off=(0, 0, 0), want=(1, 1, 1)):
    L.zr_test_describe_chain_bwd.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor,
                                             ZrTensor, ZrTensor, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_char_p, ctypes.c_size_t]
    L.zr_test_dry_run_chain_bwd.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor,
                                            ZrTensor, ZrTensor, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p]
    T = 1 << 40
    out = np.broadcast_shapes(sa, sb, sc)
    g = FakeT(T, out)
    a = FakeT(2 * T + 4 * off[0], sa, sta)
    b = FakeT(3 * T + 4 * off[1], sb)
    c = FakeT(4 * T + 4 * off[2], sc)
    grads = [k * T if w else None for k, w in zip((5, 6, 7), want)]
    buf = ctypes.create_string_buffer(8192)
    rc = L.zr_test_describe_chain_bwd(ops[op1], ops[op2], g.desc, a.desc, b.desc, c.desc, *grads,
                                      buf, 8192)
    assert rc == 0, rc
    assert L.zr_test_dry_run_chain_bwd(ops[op1], ops[op2], g.desc, a.desc, b.desc, c.desc,
                                       *grads) == 0
    return json.loads(buf.value.decode())


ops = {"add": 0, "sub": 1, "mul": 2, "div": 3}


def test_chain_backward_routes(L):
    """The two workload chains take the fused one-pass route; other layouts
    take the composed route, whose workspace holds t and grad_t."""
    d = _chain_desc(L, "mul", "add", (16, 1024, 768), (768,), (768,))
    assert d["route"] == "fused"
    (p,) = d["plans"]
    assert p["kernel"] == "chain" and p["c_scalar"] == 0 and p["inner_kept"] == 1
    assert (p["n_red"], p["ncol"]) == (16384, 768)
    d = _chain_desc(L, "add", "div", (8, 12, 1024, 1024), (1, 1, 1024, 1024), (1,))
    assert d["route"] == "fused"
    (p,) = d["plans"]
    assert p["c_scalar"] == 1 and (p["n_red"], p["ncol"]) == (96, 1024 * 1024)
    assert p["c_slots"] == p["ctas"] and d["ws_run"] >= 4 * p["ctas"]
    # The query sizes the fused route these pointers select: partials only.
    assert d["ws_query"] == d["ws_run"] < 1 << 20
    # c shaped differently from b: composed.
    d = _chain_desc(L, "mul", "add", (16, 64, 96), (96,), (64, 1))
    assert d["route"] == "composed" and d["need_t"] == 0 and d["need_gt"] == 1
    assert d["ws_run"] >= 4 * 16 * 64 * 96
    # op2 = mul with grad_c: t is needed too.
    d = _chain_desc(L, "add", "mul", (16, 64, 96), (64, 96), (16, 1, 1))
    assert d["route"] == "composed" and d["need_t"] == 1
    assert d["ws_run"] >= 2 * 4 * 16 * 64 * 96
    # a broadcast (not of the output's shape): composed.
    d = _chain_desc(L, "mul", "add", (96,), (32, 96), (32, 96))
    assert d["route"] == "composed"
    # c misaligned for 16-byte loads: composed; a gradient not requested: composed.
    d = _chain_desc(L, "mul", "add", (16, 1024, 768), (768,), (768,), off=(0, 0, 1))
    assert d["route"] == "composed"
    d = _chain_desc(L, "mul", "add", (16, 1024, 768), (768,), (768,), want=(1, 1, 0))
    assert d["route"] == "composed" and d["need_t"] == 0


def test_chain_errors_before_any_device_access(L):
    T = 1 << 40
    a, b, c = FakeT(T, (4, 8)), FakeT(2 * T, (8,)), FakeT(3 * T, (5,))
    L.zr_chain_fwd.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor, ZrTensor,
                               ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p]
    assert L.zr_chain_fwd(2, 0, a.desc, b.desc, c.desc, 4 * T, None, None) == -3
    c1 = FakeT(3 * T, (8,))
    assert L.zr_chain_fwd(9, 0, a.desc, b.desc, c1.desc, 4 * T, None, None) == -1
    # Output partially overlapping an input.
    assert L.zr_chain_fwd(2, 0, a.desc, b.desc, c1.desc, T + 4, None, None) == -5
    g = FakeT(5 * T, (4, 8))
    nbytes = ctypes.c_size_t(0)
    # A gradient overlapping an input.
    assert L.zr_chain_bwd(2, 0, g.desc, a.desc, b.desc, c1.desc, T, 6 * T, 7 * T, None,
                          ctypes.byref(nbytes), None) == -5
    # grad_out of the wrong shape.
    g2 = FakeT(5 * T, (4, 9))
    assert L.zr_chain_bwd(2, 0, g2.desc, a.desc, b.desc, c1.desc, 8 * T, 6 * T, 7 * T, None,
                          ctypes.byref(nbytes), None) == -3
    # A needed operand without data (op1 = mul: grad_a reads b).
    bn = ZrTensor(None, 1, _i64([8]), None)
    assert L.zr_chain_bwd(2, 0, g.desc, a.desc, bn, c1.desc, 8 * T, None, None, None,
                          ctypes.byref(nbytes), None) == -1
    # add then add reads no operand values: sizes alone are enough.
    an = ZrTensor(None, 2, _i64([4, 8]), None)
    cn = ZrTensor(None, 1, _i64([8]), None)
    assert L.zr_chain_bwd(0, 0, g.desc, an, bn, cn, 8 * T, 6 * T, 7 * T, None,
                          ctypes.byref(nbytes), None) == 0
    assert nbytes.value >= 4 * 32  # grad_t in the workspace


def test_backward_ex_layout_errors_and_query(L):
    """zr_binary_bwd_ex: gradients that overlap themselves or an input are
    refused before any device access; a strided or accumulated gradient adds
    its staging buffer to the workspace query."""
    from broadcast_elementwise_shape_gb300 import ZrGrad
    T = 1 << 40
    g, x, bias = FakeT(T, (64, 256)), FakeT(2 * T, (64, 256)), FakeT(3 * T, (256,))
    nb = ctypes.c_size_t(0)
    dense = ZrGrad(4 * T, None, 0)
    assert L.zr_binary_bwd_ex(0, g.desc, x.desc, bias.desc, dense, ZrGrad(5 * T, None, 0), None,
                              ctypes.byref(nb), None) == 0
    q_dense = nb.value
    # An accumulated gradient is staged too (then added in place).
    assert L.zr_binary_bwd_ex(0, g.desc, x.desc, bias.desc, dense, ZrGrad(5 * T, None, 1), None,
                              ctypes.byref(nb), None) == 0
    assert nb.value >= q_dense + 4 * 256
    # grad_a as a transposed view of a [256, 64] buffer: staged.
    st = _i64([1, 64])
    assert L.zr_binary_bwd_ex(0, g.desc, x.desc, bias.desc, ZrGrad(4 * T, st, 1),
                              ZrGrad(5 * T, None, 0), None, ctypes.byref(nb), None) == 0
    assert nb.value >= q_dense + 4 * 64 * 256
    # A gradient layout that overlaps itself.
    bad = _i64([0, 1])
    assert L.zr_binary_bwd_ex(0, g.desc, x.desc, bias.desc, ZrGrad(4 * T, bad, 0), dense, None,
                              ctypes.byref(nb), None) == -5
    # A strided gradient overlapping grad_out.
    assert L.zr_binary_bwd_ex(0, g.desc, x.desc, bias.desc, ZrGrad(T + 4, st, 0),
                              ZrGrad(5 * T, None, 0), None, ctypes.byref(nb), None) == -5
    # Negative strides are refused like any tensor's.
    neg = _i64([-1, 64])
    assert L.zr_binary_bwd_ex(0, g.desc, x.desc, bias.desc, ZrGrad(4 * T, neg, 0), dense, None,
                              ctypes.byref(nb), None) == -4


def test_float32_only_entry_points_refuse_bf16():
    """The chain and gradient-layout entry points compute on float32
    storage; the binding refuses bfloat16 tensors before any call.  The
    unary ops take either type but not a mix."""
    import torch
    h = torch.ones(4, 8, dtype=torch.bfloat16)
    v = torch.ones(8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        zr.zr_chain_fwd("mul", "add", h, v, v)
    with pytest.raises(TypeError):
        zr.zr_chain_bwd("mul", "add", h, h, v, v)
    with pytest.raises(TypeError):
        zr.zr_unary_fwd("gelu", h, out=torch.ones(4, 8))
    with pytest.raises(TypeError):
        zr.zr_unary_bwd("gelu", h, torch.ones(4, 8))
    with pytest.raises(TypeError):
        zr.zr_binary_bwd_ex("add", h, h, v, grad_a=h)
    with pytest.raises(TypeError):  # mixed element types
        zr.zr_binary_fwd("add", torch.ones(4), v[:4])


def test_describe_bwd_bf16_plans(L):
    """The element-type-aware plan description: bf16 plans take 8-wide
    vectors where the layout allows and plan the grid for the bf16 kernels'
    occupancy; an unknown element type is ZR_ERR_DTYPE."""
    L.zr_test_describe_bwd_t.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor, ZrTensor,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                         ctypes.c_size_t]
    T = 1 << 40

    def bwd(dtype, op, sa, sb):
        out = np.broadcast_shapes(sa, sb)
        g, a, b = FakeT(T, out), FakeT(2 * T, sa), FakeT(3 * T, sb)
        buf = ctypes.create_string_buffer(4096)
        rc = L.zr_test_describe_bwd_t(dtype, op, g.desc, a.desc, b.desc, 4 * T, 5 * T, buf, 4096)
        return rc, (json.loads(buf.value.decode()) if rc == 0 else None)

    # c4 in bf16: add backward with the mask reduced over 96 rows (inner kept).
    rc, d = bwd(1, 0, (8, 12, 1024, 1024), (1, 1, 1024, 1024))
    assert rc == 0
    (p,) = d["plans"]
    assert p["vec"] == 8 and p["inner_kept"] == 1 and (p["n_red"], p["ncol"]) == (96, 1024 * 1024)
    # Every reduced row in one block, 64 column lanes of 8 (each thread a
    # quarter of the rows), no partial slots.
    assert (p["tx"], p["ty"], p["rows_per_blk"], p["nslots"]) == (64, 4, 96, 1)
    assert p["ctas"] == 1024 * 1024 // 512
    # The same in float: 4-wide vectors.
    rc, d = bwd(0, 0, (8, 12, 1024, 1024), (1, 1, 1024, 1024))
    assert rc == 0 and d["plans"][0]["vec"] == 4
    # div by a scalar in bf16: full sum of g*a with grad_a written densely.
    rc, d = bwd(1, 3, (8, 12, 1024, 1024), (1,))
    assert rc == 0 and d["plans"][0]["vec"] == 8 and d["plans"][0]["dense_out"] == 1
    assert bwd(7, 0, (4, 4), (4,))[0] == -9


def _bf16_shapes(rng):
    """Shapes whose inner dim is often a multiple of 8 (16-byte bf16 vectors)."""
    n = int(rng.integers(1, 5))
    out = [int(v) for v in rng.choice([1, 2, 3, 5, 8, 16, 24], n)]
    sa = [s if rng.random() < 0.6 else 1 for s in out]
    sb = [s if rng.random() < 0.6 else 1 for s in out]
    sa[-1] = out[-1]
    return tuple(sa), tuple(sb[int(rng.integers(0, n)):])


def test_emulated_bf16_plans_match_naive(L):
    """bf16 plans (8-wide vectors where rows and 2-byte-element pointers are
    16-byte aligned, else 4 or 1): the host walk of every planned forward and
    backward kernel visits each output element once, with the offsets and
    gradient indices of the definition."""
    L.zr_test_emulate_fwd_t.argtypes = [ctypes.c_int, ZrTensor, ZrTensor, ctypes.c_void_p,
                                        ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64)]
    L.zr_test_emulate_bwd_t.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor, ZrTensor,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_int64),
                                        ctypes.POINTER(ctypes.c_int64)]
    L.zr_test_describe_bwd_t.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor, ZrTensor, ZrTensor,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_char_p,
                                         ctypes.c_size_t]
    rng = np.random.default_rng(77)
    vecs = set()
    for it in range(300):
        sa, sb = _bf16_shapes(rng)
        out_shape = np.broadcast_shapes(sa, sb)
        n_out = int(np.prod(out_shape))
        a = rand_view(rng, sa, 0x100000 + 2 * int(rng.integers(0, 8)))
        b = rand_view(rng, sb, 0x900000 + 2 * int(rng.integers(0, 2)))
        ost = dense_strides(out_shape)
        cap = n_out + 8
        rec = (ctypes.c_int64 * (3 * cap))()
        nrec = ctypes.c_int64()
        assert L.zr_test_emulate_fwd_t(1, a.desc, b.desc, 0x4000000, _i64(ost), cap, rec,
                                       ctypes.byref(nrec)) == 0
        r = np.frombuffer(rec, np.int64)[: 3 * nrec.value].reshape(-1, 3)
        assert r.shape[0] == n_out
        order = np.argsort(r[:, 0])
        np.testing.assert_array_equal(r[order, 0], np.arange(n_out))
        np.testing.assert_array_equal(r[order, 1], naive_offsets(out_shape, sa, a.strides).ravel())
        np.testing.assert_array_equal(r[order, 2], naive_offsets(out_shape, sb, b.strides).ravel())
        # Backward of mul (both operands read), both gradients requested.
        g = rand_view(rng, out_shape, 0x200000 + 2 * int(rng.integers(0, 8)))
        buf = ctypes.create_string_buffer(8192)
        assert L.zr_test_describe_bwd_t(1, 2, g.desc, a.desc, b.desc, 0x5000000, 0x6000000, buf,
                                        8192) == 0
        desc = json.loads(buf.value.decode())
        for p in desc.get("plans", []):
            vecs.add(p.get("vec"))
        rec = (ctypes.c_int64 * (7 * (2 * n_out + 8)))()
        assert L.zr_test_emulate_bwd_t(1, 2, g.desc, a.desc, b.desc, 0x5000000, 0x6000000,
                                       2 * n_out + 8, rec, ctypes.byref(nrec)) == 0
        rr = np.frombuffer(rec, np.int64)[: 7 * nrec.value].reshape(-1, 7)
        go = naive_offsets(out_shape, out_shape, g.strides).ravel()
        for pi in range(len(desc.get("plans", []))):
            rp = rr[rr[:, 0] == pi]
            assert rp.shape[0] == n_out
            np.testing.assert_array_equal(np.sort(rp[:, 1]), np.sort(go))
    assert 8 in vecs and (4 in vecs or 1 in vecs)


def test_trace_prints_the_plan_of_each_call():
    """With ZR_TRACE=1 every forward, backward, sum-to-shape and unary call
    that passes planning prints its plan to stderr (here the device checks
    then fail: no GPU, fake pointers); without it nothing is printed."""
    import subprocess
    import sys
    code = r"""
import ctypes, sys
sys.path.insert(0, %r)
import broadcast_elementwise_shape_gb300 as zr
L = zr.lib()
def T(addr, shape):
    st = []; s = 1
    for d in reversed(shape): st.insert(0, s); s *= d
    sz, stt = zr._i64(shape), zr._i64(st)
    T.keep.append((sz, stt))
    return zr.ZrTensor(addr, len(shape), sz, stt)
T.keep = []
a, b = T(1 << 40, (64, 32)), T(2 << 40, (32,))
rc1 = L.zr_binary_fwd(0, a, b, ctypes.c_void_p(3 << 40), None, None)
n = ctypes.c_size_t(1 << 20)
rc2 = L.zr_binary_bwd(2, T(4 << 40, (64, 32)), a, b, ctypes.c_void_p(5 << 40), ctypes.c_void_p(6 << 40),
                      ctypes.c_void_p(7 << 40), ctypes.byref(n), None)
L.zr_unary_fwd_t.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_float, zr.ZrTensor,
                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
L.zr_unary_bwd_t.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_float, zr.ZrTensor, zr.ZrTensor,
                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
big = (16384, 3072)
rc3 = L.zr_unary_fwd_t(1, 1, 1.0, T(8 << 40, big), ctypes.c_void_p(9 << 40), None, None)
rc4 = L.zr_unary_bwd_t(1, 1, 1.0, T(10 << 40, big), T(11 << 40, big), ctypes.c_void_p(12 << 40),
                       None, None)
print(rc1, rc2, rc3, rc4)
""" % ROOT
    env = dict(os.environ, ZR_TRACE="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("zr_trace ")]
    assert lines[0].startswith('zr_trace zr_binary_fwd {"kernel":"flat"'), lines
    assert lines[1].startswith('zr_trace zr_binary_bwd {"plans":[{"kernel":"reduce"'), lines
    json.loads(lines[1].split(" ", 2)[2])
    # bf16 GeLU on a [16384, 3072] activation: the table kernel, one CTA per SM.
    for ln, entry in ((lines[2], "zr_unary_fwd"), (lines[3], "zr_unary_bwd")):
        assert ln.startswith("zr_trace %s " % entry), lines
        d = json.loads(ln.split(" ", 2)[2])
        assert d["kernel"] == "gelu_table" and d["ctas"] == 152, d
    rcs = [int(v) for v in r.stdout.split()]
    assert all(rc in (-6, -8) for rc in rcs), rcs  # device checks fail without a GPU
    env["ZR_TRACE"] = "0"
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=120)
    assert "zr_trace" not in r.stderr


def test_emulated_eight_dim_plans_match_naive(L):
    """Rank 8 (the maximum) with broadcasting on every dim pattern: the host
    walks of the forward and backward plans visit every element once with
    the definition's offsets and gradient indices."""
    rng = np.random.default_rng(88)
    for it in range(40):
        out = [int(v) for v in rng.choice([1, 2, 3], 8)]
        sa = tuple(s if rng.random() < 0.6 else 1 for s in out)
        sb = tuple(s if rng.random() < 0.6 else 1 for s in out)
        out_shape = np.broadcast_shapes(sa, sb)
        n_out = int(np.prod(out_shape))
        a = rand_view(rng, sa, 0x100000)
        b = rand_view(rng, sb, 0x900000)
        rec = (ctypes.c_int64 * (3 * (n_out + 8)))()
        nrec = ctypes.c_int64()
        assert L.zr_test_emulate_fwd(a.desc, b.desc, 0x4000000, None, n_out + 8, rec,
                                     ctypes.byref(nrec)) == 0
        r = np.frombuffer(rec, np.int64)[: 3 * nrec.value].reshape(-1, 3)
        order = np.argsort(r[:, 0])
        np.testing.assert_array_equal(r[order, 0], np.arange(n_out))
        np.testing.assert_array_equal(r[order, 1], naive_offsets(out_shape, sa, a.strides).ravel())
        np.testing.assert_array_equal(r[order, 2], naive_offsets(out_shape, sb, b.strides).ravel())
        g = rand_view(rng, out_shape, 0x200000)
        rec = (ctypes.c_int64 * (7 * (2 * n_out + 8)))()
        assert L.zr_test_emulate_bwd(3, g.desc, a.desc, b.desc, 0x5000000, 0x6000000, 2 * n_out + 8,
                                     rec, ctypes.byref(nrec)) == 0
        rr = np.frombuffer(rec, np.int64)[: 7 * nrec.value].reshape(-1, 7)
        go = naive_offsets(out_shape, out_shape, g.strides).ravel()
        xa = grad_index(out_shape, sa).ravel()
        xb = grad_index(out_shape, sb).ravel()
        for pi in np.unique(rr[:, 0]):
            rp = rr[rr[:, 0] == pi]
            assert rp.shape[0] == n_out
            order = np.argsort(rp[:, 1])
            ref = np.argsort(go)
            np.testing.assert_array_equal(rp[order, 1], go[ref])
            x = rp[order, 4]
            if x[0] != -1:
                assert np.array_equal(x, xa[ref]) or np.array_equal(x, xb[ref])


def test_describe_unary_routes_bf16_gelu_to_its_table(L):
    """bfloat16 GeLU over a flat layout of at least 32,768 elements per SM
    (152 SMs) reads its results from a table (k_gelu_bf16, one CTA per SM,
    fewer when there are fewer passes of 1024 threads); smaller calls, float
    GeLU, scale and non-flat layouts keep the arithmetic kernels."""
    L.zr_test_describe_unary_t.argtypes = [ctypes.c_int, ctypes.c_int, ZrTensor,
                                           ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_char_p, ctypes.c_size_t]
    T = 1 << 40

    def desc(dtype, op, shape, strides=None, bwd=False, out_strides=None):
        x = FakeT(T, shape, strides)
        g = FakeT(2 * T, shape, strides)
        ost = _i64(out_strides) if out_strides is not None else None
        buf = ctypes.create_string_buffer(4096)
        if bwd:
            rc = L.zr_test_describe_unary_t(dtype, op, g.desc, ctypes.addressof(x.desc), 3 * T,
                                            ctypes.cast(ost, ctypes.c_void_p) if ost else None,
                                            buf, 4096)
        else:
            rc = L.zr_test_describe_unary_t(dtype, op, x.desc, None, 3 * T,
                                            ctypes.cast(ost, ctypes.c_void_p) if ost else None,
                                            buf, 4096)
        assert rc == 0, rc
        return json.loads(buf.value.decode())

    BF16, F32, SCALE, GELU = 1, 0, 0, 1
    for bwd in (False, True):
        d = desc(BF16, GELU, (16384, 3072), bwd=bwd)  # a [16384, 3072] activation
        assert d["kernel"] == "gelu_table" and d["vec"] == 8 and d["ctas"] == 152, d
        assert desc(F32, GELU, (16384, 3072), bwd=bwd)["kernel"] == "flat"
        assert desc(BF16, SCALE, (16384, 3072), bwd=bwd)["kernel"] == "flat"
        # Just below and at the size limit.
        assert desc(BF16, GELU, (152 * 32768 - 8,), bwd=bwd)["kernel"] == "flat"
        assert desc(BF16, GELU, (152 * 32768,), bwd=bwd)["kernel"] == "gelu_table"
    # Odd sizes take 1-element items, row-strided views rows of 8.
    d = desc(BF16, GELU, (152 * 32768 + 1,))
    assert d["kernel"] == "gelu_table" and d["vec"] == 1 and d["ctas"] == 152
    d = desc(BF16, GELU, (2048, 8192), strides=(8200, 1))
    assert d["kernel"] == "gelu_table" and d["vec"] == 8 and d["row_dims"] == 1
    # A layout that does not flatten to two dims keeps the tiled kernel.
    d = desc(BF16, GELU, (64, 64, 4096), strides=(64 * 4104, 4104, 1),
             out_strides=(64 * 4096 + 8, 4096, 1))
    assert d["kernel"] == "elementwise"
