"""CPU oracle for broadcasting elementwise binary ops — TEST INFRASTRUCTURE.

Plain C++ (``zr_oracle.cpp``, single thread, binary64 accumulation, built with
``-O2 -ffp-contract=off``), wrapped here with ctypes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The product library never does, and the
two share no code.

What it computes follows the "Zero" book (ismantic.github.io/zero):
Operator page, sections "逐元素算子" (elementwise ops) and "广播"
(broadcasting, sum back to shape); Tensor page, section "形状与步长"
(shape and strides); GPU page, section "OpAdd" (add's local derivative).
sub/div backward use the calculus rules (g, -g) and (g/b, -g*a/b^2), which
the pages leave unstated.  Two-op chains (a op1 b) op2 c are the composition
of two of these operators (Operator page, section 融合; Autograd page,
section 链式法则).

Pins (tests/test_oracle_pins.py, all CPU): the pages' printed broadcast,
stride and transposed-view examples, the worked gradient z = x*y + x at
x=3, y=2, NumPy broadcasting and float32 arithmetic, float64 central
finite differences, closed forms of sum-to-shape, and scatter-vs-gather
agreement; the chains by the same worked gradient (z = x*y + x is the chain
(x mul y) add x), NumPy float32 two-step forwards, closed forms of the affine
and scaled-mask chains, and float64 finite differences of all 16 op pairs.
Every function here is pinned by at least one of them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zr_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

ADD, SUB, MUL, DIV = 0, 1, 2, 3
OPS = {"add": ADD, "sub": SUB, "mul": MUL, "div": DIV}


def build(force: bool = False) -> str:
    """Compile the oracle to ``oracle/_build/liboracle.so`` (g++, -O2, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.{os.getpid()}.tmp"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            vp = ctypes.c_void_p
            ci = ctypes.c_int
            ten = [vp, ci, i64p, i64p]
            _lib.orc_contiguous_strides.argtypes = [ci, i64p, i64p]
            _lib.orc_broadcast_shape.argtypes = [ci, i64p, ci, i64p, ctypes.POINTER(ci), i64p]
            _lib.orc_binary_fwd.argtypes = [ci] + ten + ten + [vp]
            _lib.orc_binary_fwd_at.argtypes = [ci] + ten + ten + [ctypes.c_int64, i64p, vp]
            _lib.orc_binary_bwd.argtypes = [ci] + ten + ten + ten + [vp, vp, vp, vp]
            _lib.orc_binary_bwd_at.argtypes = [ci, ci] + ten + ten + ten + [ctypes.c_int64, i64p, vp, vp]
            _lib.orc_sum_to_shape.argtypes = ten + [ci, i64p, vp, vp]
            _lib.orc_sum_to_shape_at.argtypes = ten + [ci, i64p, ctypes.c_int64, i64p, vp, vp]
            _lib.orc_round_bf16.argtypes = [vp, ctypes.c_int64, vp]
            _lib.orc_round_bf16.restype = ci
            _lib.orc_unary_fwd.argtypes = [ci, ctypes.c_float] + ten + [vp]
            _lib.orc_unary_bwd.argtypes = [ci, ctypes.c_float] + ten + [vp, i64p, vp, vp]
            for f in ("orc_unary_fwd", "orc_unary_bwd"):
                getattr(_lib, f).restype = ci
            for f in ("orc_contiguous_strides", "orc_broadcast_shape", "orc_binary_fwd",
                      "orc_binary_fwd_at", "orc_binary_bwd", "orc_binary_bwd_at",
                      "orc_sum_to_shape", "orc_sum_to_shape_at"):
                getattr(_lib, f).restype = ci
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: oracle returned {rc}")


def _i64(seq):
    arr = (ctypes.c_int64 * max(1, len(seq)))(*[int(s) for s in seq])
    return arr


class _T:
    """A strided float32 host view: (base pointer, sizes, element strides).

    Accepts a torch CPU tensor (any strides, storage offset included in
    ``data_ptr()``), a NumPy array, or ``None`` with an explicit shape (for
    operands whose data the op does not read).
    """

    def __init__(self, x, shape=None):
        self.keep = x
        if x is None:
            self.ptr = None
            self.sizes = list(shape)
            self.strides = None
        elif hasattr(x, "data_ptr"):  # torch tensor
            import torch
            if x.dtype != torch.float32 or x.device.type != "cpu":
                raise TypeError("oracle takes float32 CPU tensors")
            self.ptr = x.data_ptr() if x.numel() > 0 else None
            self.sizes = list(x.shape)
            self.strides = list(x.stride())
        else:
            x = np.asarray(x)
            if x.dtype != np.float32:
                raise TypeError("oracle takes float32 arrays")
            self.keep = x
            self.ptr = x.ctypes.data if x.size > 0 else None
            self.sizes = list(x.shape)
            self.strides = [s // 4 for s in x.strides]
        self._sz = _i64(self.sizes)
        self._st = _i64(self.strides) if self.strides is not None else None

    def args(self):
        return [self.ptr, len(self.sizes), self._sz, self._st]


def contiguous_strides(shape):
    lib = _load()
    out = (ctypes.c_int64 * max(1, len(shape)))()
    _check(lib.orc_contiguous_strides(len(shape), _i64(shape), out), "contiguous_strides")
    return tuple(out[i] for i in range(len(shape)))


def broadcast_shape(shape_a, shape_b):
    """Broadcast shape, or raise OracleError if incompatible."""
    lib = _load()
    nd = ctypes.c_int(0)
    out = (ctypes.c_int64 * 8)()
    _check(lib.orc_broadcast_shape(len(shape_a), _i64(shape_a), len(shape_b), _i64(shape_b),
                                   ctypes.byref(nd), out), "broadcast_shape")
    return tuple(out[i] for i in range(nd.value))


def binary_fwd(op, a, b):
    """out = a op b, dense row-major float32 of the broadcast shape."""
    lib = _load()
    op = OPS.get(op, op)
    ta, tb = _T(a), _T(b)
    shape = broadcast_shape(ta.sizes, tb.sizes)
    out = np.empty(shape, dtype=np.float32)
    _check(lib.orc_binary_fwd(op, *ta.args(), *tb.args(), out.ctypes.data if out.size else None),
           "binary_fwd")
    return out


def binary_fwd_at(op, a, b, idx):
    """Forward values at output linear indices ``idx`` (row-major)."""
    lib = _load()
    op = OPS.get(op, op)
    ta, tb = _T(a), _T(b)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = np.empty(idx.shape, dtype=np.float32)
    _check(lib.orc_binary_fwd_at(op, *ta.args(), *tb.args(), idx.size,
                                 idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 vals.ctypes.data if vals.size else None), "binary_fwd_at")
    return vals


def binary_bwd(op, g, a, b, want_a=True, want_b=True, shape_a=None, shape_b=None):
    """(grad_a, grad_b, abs_a, abs_b): gradients dense in each input's shape,
    plus sum|term| per gradient element (float64).  Pass ``a``/``b`` as None
    with ``shape_a``/``shape_b`` when the op does not read them."""
    lib = _load()
    op = OPS.get(op, op)
    tg, ta, tb = _T(g), _T(a, shape_a), _T(b, shape_b)
    ga = np.empty(ta.sizes, dtype=np.float32) if want_a else None
    gb = np.empty(tb.sizes, dtype=np.float32) if want_b else None
    sa = np.empty(ta.sizes, dtype=np.float64) if want_a else None
    sb = np.empty(tb.sizes, dtype=np.float64) if want_b else None

    def p(x):
        return None if x is None else x.ctypes.data

    _check(lib.orc_binary_bwd(op, *tg.args(), *ta.args(), *tb.args(), p(ga), p(gb), p(sa), p(sb)),
           "binary_bwd")
    return ga, gb, sa, sb


def binary_bwd_at(op, which, g, a, b, idx, shape_a=None, shape_b=None):
    """Gradient values (and sum|term|) of grad_a (which=0) or grad_b (which=1)
    at linear indices ``idx`` of that input's dense row-major shape."""
    lib = _load()
    op = OPS.get(op, op)
    tg, ta, tb = _T(g), _T(a, shape_a), _T(b, shape_b)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = np.empty(idx.shape, dtype=np.float32)
    sabs = np.empty(idx.shape, dtype=np.float64)
    _check(lib.orc_binary_bwd_at(op, which, *tg.args(), *ta.args(), *tb.args(), idx.size,
                                 idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 vals.ctypes.data if vals.size else None,
                                 sabs.ctypes.data if sabs.size else None), "binary_bwd_at")
    return vals, sabs


def sum_to_shape(x, shape):
    """(out, abs): binary64 sums of x down to ``shape`` rounded once, and sum|x|."""
    lib = _load()
    tx = _T(x)
    out = np.empty(shape, dtype=np.float32)
    sabs = np.empty(shape, dtype=np.float64)
    _check(lib.orc_sum_to_shape(*tx.args(), len(shape), _i64(shape),
                                out.ctypes.data if out.size else None,
                                sabs.ctypes.data if sabs.size else None), "sum_to_shape")
    return out, sabs


def sum_to_shape_at(x, shape, idx):
    lib = _load()
    tx = _T(x)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = np.empty(idx.shape, dtype=np.float32)
    sabs = np.empty(idx.shape, dtype=np.float64)
    _check(lib.orc_sum_to_shape_at(*tx.args(), len(shape), _i64(shape), idx.size,
                                   idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   vals.ctypes.data if vals.size else None,
                                   sabs.ctypes.data if sabs.size else None), "sum_to_shape_at")
    return vals, sabs


# ---------------------------------------------------------------- two-op chains
#
# out = (a op1 b) op2 c: two of the operators above applied in sequence, each
# rounded to binary32 — the fused forms the Operator page's section 融合
# (fusion) motivates (fewer launches, no intermediate round trip through
# memory), which keep the operators' mathematical definition.  The oracle
# is that definition: the two forward ops one after the other, and the
# backward by the chain rule (Autograd page, section 链式法则): op2's local
# rules give grad_t and grad_c, op1's rules applied to grad_t give grad_a and
# grad_b.  t and grad_t are rounded to binary32 in between, as the unfused
# ops would store them.

def chain_fwd(op1, op2, a, b, c):
    """out = (a op1 b) op2 c, dense float32 of the broadcast of all three."""
    t = binary_fwd(op1, a, b)
    return binary_fwd(op2, t, c)


def chain_bwd(op1, op2, g, a, b, c):
    """(grad_a, grad_b, grad_c, abs_a, abs_b, abs_c) of out = (a op1 b) op2 c
    given grad_out g; abs_* are sum|term| per gradient element (float64),
    with the terms of grad_a and grad_b taken from the binary32 grad_t."""
    t = binary_fwd(op1, a, b)
    gt, gc, _, sc = binary_bwd(op2, g, t, c)
    ga, gb, sa, sb = binary_bwd(op1, gt, a, b)
    return ga, gb, gc, sa, sb, sc


def chain_bwd_at(op1, op2, which, g, a, b, c, idx):
    """Values (and sum|term|) of grad_a (which=0), grad_b (1) or grad_c (2)
    at linear indices ``idx`` of that input's dense row-major shape."""
    t = binary_fwd(op1, a, b)
    if which == 2:
        return binary_bwd_at(op2, 1, g, t, c, idx)
    gt, _, _, _ = binary_bwd(op2, g, t, c, want_b=False)
    return binary_bwd_at(op1, which, gt, a, b, idx)


# ---------------------------------------------------------------- accumulation

def accumulate(old, new):
    """AccumulateGrad (Autograd page, section 反向传播): a gradient slot that
    already holds a value gets the new gradient added in place — one binary32
    addition per element, so a tensor reached by several paths receives the
    sum of their gradients."""
    return (np.asarray(old, dtype=np.float32) + np.asarray(new, dtype=np.float32)).astype(np.float32)



# ---------------------------------------------------------------- unary ops
#
# GPU page, section 逐元素运算: GeLU and gradient scaling are elementwise.
# scale: alpha * x (one binary32 multiply); GeLU: the exact x * Phi(x) (the
# pages give no formula), evaluated in binary64 and rounded once.

UNARY = {"scale": 0, "gelu": 1}


def unary_fwd(op, x, alpha=1.0):
    """out = op(x), dense float32 of x's shape."""
    lib = _load()
    tx = _T(x)
    out = np.empty(tx.sizes, dtype=np.float32)
    _check(lib.orc_unary_fwd(UNARY.get(op, op), alpha, *tx.args(), out.ctypes.data if out.size else None),
           "unary_fwd")
    return out


def unary_bwd(op, g, x, alpha=1.0):
    """(grad_x, mag): grad_x = g * op'(x) dense float32; mag the size of the
    terms before rounding (|g| (Phi(x) + |x| phi(x)) for GeLU, float64)."""
    lib = _load()
    tg = _T(g)
    tx = _T(x) if x is not None else _T(None, tg.sizes)
    if tx.sizes != tg.sizes:
        raise OracleError("unary_bwd: g and x differ in shape")
    out = np.empty(tg.sizes, dtype=np.float32)
    mag = np.empty(tg.sizes, dtype=np.float64)
    _check(lib.orc_unary_bwd(UNARY.get(op, op), alpha, *tg.args(), tx.ptr, tx._st,
                             out.ctypes.data if out.size else None,
                             mag.ctypes.data if mag.size else None), "unary_bwd")
    return out, mag



# ---------------------------------------------------------------- bf16 storage
#
# A bfloat16 operator reads bf16 inputs (exact binary32 values), computes as
# the binary32 operator does, and stores each result rounded once to bf16.
# For one +, -, *, / the binary32 result rounded to bf16 equals the exact
# result rounded to bf16 (binary32 has 24 >= 2 * 8 + 2 significand bits, so
# the double rounding is innocuous; Figueroa), so bf16 outputs of the
# forward and of one-operation gradients are fixed bit for bit; summed
# gradients are the binary64 sums rounded to binary32 and then to bf16.

def round_bf16(x):
    """Round float32 values to the nearest bfloat16 (ties to even), returned
    as the float32 values they denote."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    _check(lib.orc_round_bf16(x.ctypes.data if x.size else None, x.size,
                              out.ctypes.data if out.size else None), "round_bf16")
    return out
