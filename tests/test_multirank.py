"""Multi-process host logic of bench.py on CPU: two gloo ranks.

Systems are independent, so the GPU path shards by batch with no collective on
the data path; the ranks only meet at barriers and in a max over their timings.
This test runs that host logic with world_size 2 on the CPU."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    d = bench.Dist(world)
    try:
        d.barrier()
        m = d.max(float(10 * rank + 3))
        res = {"rank": rank, "max": m, "weak": bench.shard(65536, world, rank, weak=True),
               "strong": bench.shard(65537, world, rank, weak=False)}
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump(res, fh)
        d.barrier()
    finally:
        d.close()


def test_two_gloo_ranks_barrier_max_and_shard(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(2)]
    assert r[0]["max"] == r[1]["max"] == 13.0
    assert r[0]["weak"] == r[1]["weak"] == 65536          # weak scaling: full batch per GPU
    assert r[0]["strong"] + r[1]["strong"] == 65537       # strong split covers every system once
    assert abs(r[0]["strong"] - r[1]["strong"]) <= 1


def _ref_main(rank, world, port, out_dir):
    import contextlib
    import io
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "small", "--steps", "2",
                         "--warmup", "3", "--gpus", str(world)])
    with open(os.path.join(out_dir, f"ref{rank}.txt"), "w") as fh:
        fh.write(f"{rc}\n{buf.getvalue()}")


def test_reference_arm_prints_once_from_rank0(tmp_path):
    pytest.importorskip("numpy")
    port = _free_port()
    mp.start_processes(_ref_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    out0 = open(tmp_path / "ref0.txt").read().splitlines()
    out1 = open(tmp_path / "ref1.txt").read().splitlines()
    assert out0[0] == "0" and out1[0] == "0"
    lines0 = [l for l in out0[1:] if l.strip()]
    assert len(lines0) == 1 and [l for l in out1[1:] if l.strip()] == []
    rec = json.loads(lines0[0])
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
