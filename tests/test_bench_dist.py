"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each rank verifies its own batch (weak scaling): the ranks get different
seeded inputs, the step time is the max over ranks and the throughput the sum
of the units all ranks processed; there is no collective on the data path.
"""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    from speculative_decoding_verification_64_gb300 import workloads as W
    d = bench.Dist()
    d.init("gloo")
    mx = d.max(float(rank + 1) * 1.5, "cpu")
    sm = d.sum(float(rank + 1), "cpu")
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=2, V=300, seed_offset=1000 * d.rank)
    d.barrier()
    # the reference arm runs on rank 0 only; the other ranks return without work
    if rank == 1:
        import io
        import contextlib
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1"]), d)
        ref_out = buf.getvalue()
    else:
        ref_out = None
    queue.put((rank, mx, sm, w.uniforms.tobytes(), w.logits.tobytes(), ref_out))
    d.close()


def test_two_rank_timing_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r = q.get(timeout=300)
        res[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert res[r][1] == 3.0          # max over ranks
        assert res[r][2] == 3.0          # sum over ranks
    assert res[0][3] != res[1][3]        # each rank has its own uniforms
    assert res[0][4] != res[1][4]        # and its own logits
    assert res[1][5] == ""               # rank 1 printed nothing in the reference arm


def test_algorithmic_bytes_counts_every_logit_once():
    import bench
    from speculative_decoding_verification_64_gb300 import workloads as W
    w = W.make_workload("linear_b256_g8_v128256_bf16", B=3, V=1000)
    ab = bench.algorithmic_bytes(w, 2.0)
    assert ab["logits"] == 3 * 9 * 1000 * 2
    assert ab["q_rows"] == 2 * 1000 * 2
    assert ab["total"] > ab["logits"] + ab["q_rows"]
    assert np.isclose(ab["total"], ab["logits"] + ab["q_rows"] + ab["small"])


def test_reference_arm_prints_the_contract_line(capsys):
    """The reference arm (the float64 oracle on the host cores) prints one JSON
    line with the keys the benchmark contract names, on the same metric."""
    import json
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "3",
                             "--batch", "3", "--vocab", "300"])
    bench.run_reference(args, bench.Dist())
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["unit"] == "positions/s"
    assert "workload" in d["config"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in d["cpu_baseline"], key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
