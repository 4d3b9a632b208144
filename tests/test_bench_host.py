"""Host logic of bench.py that needs no GPU: the per-op copy schedule of the
end-to-end measurement reads and writes exactly the tensors each step names,
and each upload of a pipelined step waits for the previous step's last
reader of that buffer."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _allocated(step):
    """Outputs bench.Suite allocates for a step."""
    if step[0] in ("fwd", "cfwd", "ufwd", "ubwd"):
        return [step[-1]]
    return list(step[7:10] if step[0] == "cbwd" else step[5:7])


def test_step_io_covers_every_workload_step():
    for name, steps in workloads.STEPS.items():
        host = workloads.make_inputs(name, **workloads.small_dims(name))
        known = set(host)
        for step in steps:
            reads, writes = bench.step_io(step)
            names = [x for x in step[1:] if isinstance(x, str) and x not in
                     ("add", "sub", "mul", "div", "gelu", "scale")]
            assert sorted(reads + writes) == sorted(names), (name, step)
            assert writes == _allocated(step), (name, step)
            # Every operand is a host input or the output of an earlier step,
            # so uploading inputs before their first reader is a valid order.
            assert all(k in known for k in reads), (name, step)
            known.update(writes)


def test_oracle_pool_runs_every_process_over_the_whole_sample():
    """The all-cores CPU baseline: each process computes the complete sample,
    so one pass moves processes x the sample's bytes."""
    one_bytes = sum(bench.op_bytes(s, bench.shape_table("c1", workloads.make_inputs("c1"))[0])
                    for s in workloads.STEPS["c1"])
    pool = bench.OraclePool(["c1"], procs=2)
    try:
        span, nbytes, elems = pool.run()
    finally:
        pool.close()
    assert pool.n == 2 and nbytes == 2 * one_bytes and span > 0
    assert all(not p.is_alive() for p in pool.procs)


def test_kernel_hash_covers_code_only():
    """Comments and blank lines do not change the key of the measured traffic;
    code does."""
    a = "int f() {  // one\n  /* two\n three */ return 1;\n\n}\n"
    b = "int f() {\n  return 1;\n}\n"
    c = "int f() {\n  return 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b) != bench._code_only(c)
    assert bench.kernel_hash() == bench.kernel_hash()


def test_oracle_pool_takes_reduced_size_workloads():
    """The host baseline also times the strided workloads at reduced sizes:
    (name, size overrides) pairs are drawn at those sizes, and the baseline's
    default sample names c5a and c5b."""
    sample = [("c5a", dict(P=2, M=8, Q=16)), ("c5b", workloads.small_dims("c5b"))]
    want = 0
    for name, dims in sample:
        sizes = bench.shape_table(name, workloads.make_inputs(name, **dims))[0]
        want += sum(bench.op_bytes(s, sizes) for s in workloads.STEPS[name])
    pool = bench.OraclePool(sample, procs=1)
    try:
        span, nbytes, elems = pool.run()
    finally:
        pool.close()
    assert nbytes == want and span > 0
    labels = bench.sample_label(bench.CPU_SAMPLE)
    assert any(x.startswith("c5a[") for x in labels) and any(x.startswith("c5b[") for x in labels)
    assert bench.sample_label(sample)[0] == "c5a[P=2,M=8,Q=16]"


def test_pipelined_uploads_wait_for_the_last_reader():
    """Brute force over every workload: the step an upload must wait for is
    the last one that reads the buffer, so no later step of the previous
    iteration reads it after the next iteration overwrites it."""
    for name, steps in workloads.STEPS.items():
        last = bench.last_readers(steps)
        for k, i in last.items():
            readers = [j for j, st in enumerate(steps) if k in bench.step_io(st)[0]]
            assert readers and i == readers[-1], (name, k)
            assert all(k not in bench.step_io(st)[0] for st in steps[i + 1:]), (name, k)
    # c3: x is read by the forward mul and again by the backward mul.
    assert bench.last_readers(workloads.STEPS["c3"])["x"] == 3
