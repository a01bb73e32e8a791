"""The N > 1 path on CPU: gloo ranks, world size 2.

Sequences are independent, so the batch shards across ranks with no exchange on
the data path; ranks only max-reduce their elapsed time (weak scaling).  The
oracle stands in for each rank's GPU here (no GPU on this machine): the sharded
results, gathered afterwards, must equal one unsharded run.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_path):
    sys.path.insert(0, ROOT)
    import oracle
    import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = workloads.make("c3", B=8, V=3001)
    prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
    shard = np.array_split(np.arange(w["B"]), world)[rank]
    import time
    t0 = time.perf_counter()
    d = oracle.sample_draft(w["draft"][shard], w["u_draft"][shard], **prm)["tokens"]
    r = oracle.verify(w["target"][shard], w["draft"][shard], d, w["u_verify"][shard], **prm)
    el = torch.tensor([time.perf_counter() - t0], dtype=torch.float64)
    dist.all_reduce(el, op=dist.ReduceOp.MAX)  # the only cross-rank operation of a step
    parts = [None] * world
    dist.all_gather_object(parts, (shard.tolist(), r["tokens"].tolist(), r["num_accepted"].tolist()))
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump({"parts": parts, "max_elapsed": float(el.item())}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_without_exchange(tmp_path):
    import oracle
    import workloads
    oracle.build()
    out = str(tmp_path / "res.json")
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    res = json.load(open(out))
    w = workloads.make("c3", B=8, V=3001)
    prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
    d = oracle.sample_draft(w["draft"], w["u_draft"], **prm)["tokens"]
    ref = oracle.verify(w["target"], w["draft"], d, w["u_verify"], **prm)
    toks = np.zeros_like(ref["tokens"])
    n = np.zeros_like(ref["num_accepted"])
    seen = []
    for shard, t, nn in res["parts"]:
        toks[shard] = t
        n[shard] = nn
        seen += shard
    assert sorted(seen) == list(range(w["B"]))
    np.testing.assert_array_equal(toks, ref["tokens"])
    np.testing.assert_array_equal(n, ref["num_accepted"])
    assert res["max_elapsed"] > 0


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--workload", "c1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0
