"""The N > 1 path of the bench on CPU: two ranks over gloo (the path has no
exchange step, so N GPUs run N independent replicas; only the timing and the
reporting meet across ranks).

* The timings every rank reports are each value's maximum over the ranks (the
  slowest replica), and the whole-job value is all ranks' units over that time.
* Under N ranks the reference arm runs on rank 0 alone; the other ranks exit
  without work or output.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout
from types import SimpleNamespace

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist            # noqa: E402
import torch.multiprocessing as mp          # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured (r + 1) * 10 ms, (r + 1) * 20 ms, 7 ms
    got = bench.max_over_ranks([(rank + 1) * 10.0, (rank + 1) * 20.0, 7.0], dist, "cpu")
    value = bench.replica_value(world, 256 * 100, got[0])
    args = SimpleNamespace(cpu_seqs=1, cpu_steps=1, steps=1, warmup=0)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, rank, world)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "value": value, "stdout": buf.getvalue()}, f)


def test_two_ranks_over_gloo(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == [20.0, 40.0, 7.0]                 # the slowest rank's times on every rank
        assert r["value"] == pytest.approx(2 * 256 * 100 / 0.020)
    assert res[1]["stdout"] == ""                            # rank 1: no work, no line
    line = json.loads(res[0]["stdout"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_single_process_passes_values_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]
    assert bench.replica_value(1, 1000, 500.0) == pytest.approx(2000.0)


def test_memory_report_of_the_bench_line():
    """The bench line's memory report: per-sequence cache bytes of each replay
    variant against the conventional state, and sequences in 100 GiB for 24 layers."""
    sys.path.insert(0, ROOT)
    import bench
    m = bench.memory_report(128, 64, 128, 8, 16)
    json.dumps(m)                                            # serialisable
    assert m["fp32"]["bytes_per_seq_layer"] == 4194304 + 16 * 20992 + 12
    assert m["conventional"] == {"bytes_per_seq_layer": 4194304, "sequences": 1066}
    assert m["fp32"]["sequences"] == 987 and m["fp16_nvfp4_copy"]["sequences"] == 1464
    assert m["fp32_fp8_copy"]["bytes_per_seq_layer"] == m["fp32"]["bytes_per_seq_layer"] + 1081344


def test_period_weighted_step():
    """The figure beside the headline: one flush period from the per-step medians."""
    sys.path.insert(0, ROOT)
    import bench
    split = {"nonflush": [170.0, 168.0, 172.0], "flush": [370.0]}
    pw = bench.period_weighted(split, 16, 256)
    assert pw["us_per_step"] == pytest.approx((15 * 170.0 + 370.0) / 16)
    assert pw["value"] == pytest.approx(256 / (pw["us_per_step"] * 1e-6), rel=1e-6)
    assert bench.period_weighted({"nonflush": [1.0], "flush": []}, 16, 256) is None


def test_all_cores_oracle_baseline():
    """The oracle on every host core: spawned processes on their own sequences;
    the rate counts every process's sequence-steps over the slowest one."""
    sys.path.insert(0, ROOT)
    import bench
    from ssm_decode_state_gb300 import inputs as gen
    shape = gen.Mamba2Shape(8, 4, 16, 16, 1, 16)
    rate, el, cores, sample = bench.oracle_rate_all_cores(shape, 5, 2, 3, cores=2)
    assert cores == 2 and el > 0 and rate == pytest.approx(2 * 2 * 3 / el)
    assert "2 processes" in sample
