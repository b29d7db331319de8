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
