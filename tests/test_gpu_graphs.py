"""The C ABI inside CUDA graphs.  The library never allocates, synchronises
or reads device memory on the host, and every launch goes to the caller's
stream, so a whole training-style step of its calls can be captured once
(stream capture) and replayed with new values in the same buffers.  The
replayed results must match the oracle on the new values exactly as an
eager call does (bit-exact forwards and single-operation gradients, summed
gradients within 1e-5 * sum|terms|).  Launches with programmatic dependent
launch become programmatic graph edges; cluster launches keep their
cluster shape."""
import numpy as np
import pytest
import torch

import broadcast_elementwise_shape_gb300 as zr
import oracle
import workloads
from parity import bitexact, within

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zr.build()
    zr.lib()


def _ws(op, g, a, b, ga, gb):
    """Workspace for a backward call, allocated before capture (a query
    launches nothing)."""
    import ctypes
    dg, k1 = zr._desc(g)
    da, k2 = zr._desc(a)
    db, k3 = zr._desc(b)
    n = ctypes.c_size_t(0)
    rc = zr.lib().zr_binary_bwd_t(zr.ZR_F32, zr.OPS[op], dg, da, db, ga.data_ptr(), gb.data_ptr(),
                                  None, ctypes.byref(n), None)
    assert rc == 0
    return torch.empty(max(16, n.value), dtype=torch.uint8, device="cuda")


def _to_dev(v):
    """Device copy of a host view: the whole storage, same strides."""
    st = v.untyped_storage()
    flat = torch.empty(0, dtype=v.dtype).set_(st, 0, (st.nbytes() // 4,), (1,))
    return flat.cuda().as_strided(v.shape, v.stride(), v.storage_offset())


def _check_bwd(op, g, a, b, ga, gb, what):
    ra, rb, sa, sb = oracle.binary_bwd(op, g, a, b)
    for w, (got, ref, sabs, shape) in enumerate(((ga, ra, sa, a.shape), (gb, rb, sb, b.shape))):
        n_in = int(np.prod(shape))
        single = n_in == g.numel() and not (op == "div" and w == 1)
        if single:
            bitexact(got.cpu().numpy(), ref, f"{what} grad_{'ab'[w]}")
        else:
            within(got.cpu().numpy(), ref, sabs, f"{what} grad_{'ab'[w]}")


@pytest.mark.parametrize("name", ["c3", "c5a", "c5b"])
def test_step_captured_once_and_replayed(name):
    dims = workloads.small_dims(name)
    steps = workloads.STEPS[name]
    host = workloads.make_inputs(name, **dims)
    dev = {k: _to_dev(v) for k, v in host.items()}
    # Outputs and workspaces exist before capture; the graph reuses them.
    env = dict(dev)
    ws = {}
    for st in steps:
        if st[0] == "fwd":
            _, op, an, bn, on = st
            env[on] = torch.empty(torch.broadcast_shapes(env[an].shape, env[bn].shape), device="cuda")
        else:
            _, op, gn, an, bn, gan, gbn = st
            env[gan] = torch.empty(env[an].shape, device="cuda")
            env[gbn] = torch.empty(env[bn].shape, device="cuda")
            ws[st] = _ws(op, env[gn], env[an], env[bn], env[gan], env[gbn])

    def step():
        for st in steps:
            if st[0] == "fwd":
                _, op, an, bn, on = st
                zr.zr_binary_fwd(op, env[an], env[bn], out=env[on])
            else:
                _, op, gn, an, bn, gan, gbn = st
                zr.zr_binary_bwd(op, env[gn], env[an], env[bn], grad_a=env[gan], grad_b=env[gbn],
                                 workspace=ws[st])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed in (2101, 2102):
        new = workloads.make_inputs(name, seed=seed, **dims)
        for k, v in new.items():
            # Same storage, same layout: copy the whole storage of each view.
            dst = dev[k]
            st_d = dst.untyped_storage()
            st_h = v.untyped_storage()
            torch.empty(0, device="cuda").set_(st_d, 0, (st_d.nbytes() // 4,), (1,)).copy_(
                torch.empty(0).set_(st_h, 0, (st_h.nbytes() // 4,), (1,)))
        graph.replay()
        torch.cuda.synchronize()
        ref = dict(new)
        for st in steps:
            if st[0] == "fwd":
                _, op, an, bn, on = st
                ref[on] = torch.from_numpy(oracle.binary_fwd(op, ref[an], ref[bn]))
                bitexact(env[on].cpu().numpy(), ref[on].numpy(), f"{name} seed {seed} {op} fwd")
            else:
                _, op, gn, an, bn, gan, gbn = st
                # The oracle's backward reads the values the GPU step read.
                g_in = ref[gn] if gn in ref else torch.from_numpy(env[gn].cpu().numpy())
                _check_bwd(op, g_in, ref[an], ref[bn], env[gan], env[gbn],
                           f"{name} seed {seed} {op} bwd")
                ref[gan] = torch.from_numpy(env[gan].cpu().numpy())
                ref[gbn] = torch.from_numpy(env[gbn].cpu().numpy())
