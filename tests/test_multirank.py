"""N > 1 host logic of bench.py on CPU: world-size-2 gloo ranks agree on the
max step time, the whole-job value sums every rank's bytes, and only rank 0
reports (the reference arm's other ranks exit without work)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist = bench.init_dist(world, "gloo")
    ws_, r, _ = bench.dist_env()
    mx = bench.reduce_max(10.0 + 5.0 * rank, dist)          # rank 1 is the slow one
    val = bench.weak_scaling_value(1e9, 100, mx, ws_)
    args = type("A", (), dict(steps=1, warmup=0, workload="q6k_512x2048"))()
    ref = bench.bench_reference(args, ws_, r) if r != 0 else "rank0"
    out.put((r, mx, val, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, mx0, v0, ref0), (r1, mx1, v1, ref1) = res
    assert mx0 == mx1 == 15.0                                 # max over ranks
    assert v0 == pytest.approx(2 * 1e9 * 100 / 15e-3 / 1e9)   # both ranks' bytes / slowest time
    assert ref1 is None                                       # non-zero ranks report nothing


@pytest.mark.parametrize("act,dtype", [("q8", "i8"), ("f32", "f32")])
def test_reference_arm_line(act, dtype):
    """The reference arm (the oracle on the host, one rank): its JSON line
    carries the contract's keys, a zero-copy e2e and the oracle baseline."""
    import bench
    args = type("A", (), dict(steps=1, warmup=3, workload="q6k_512x2048", tokens=1, act=act))()
    line = bench.bench_reference(args, 1, 0)
    assert line["impl"] == "reference" and line["dtype"] == dtype
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert act in line["config"]["sample"]
