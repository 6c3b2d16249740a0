"""Host-side logic of bench.py: the multi-rank timing aggregation (gloo,
world size 2, on the CPU) and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    bench.init_dist(world, "gloo")
    t = [1.5, 2.0][rank]                     # rank 1 is the slower one
    tmax = bench.reduce_max(t, world)
    gbs = bench.job_throughput(1e9, world, tmax, 10)
    bench.barrier(world)
    q.put((rank, tmax, gbs))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29511
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, tmax, gbs in res:
        assert tmax == 2.0                       # the slowest rank sets the job time
        assert gbs == pytest.approx(1e9 * 2 * 10 / 2.0 / 1e9)   # both ranks' bytes


def test_step_bytes_formula():
    sys.path.insert(0, ROOT)
    import bench
    from static_kv_cache_gb300 import synth
    w = synth.WORKLOADS["llama2_70b_b1"]
    b = bench.step_bytes(w, [32768])
    assert b["attn"] == 1073741824 + 2 * 64 * 128 * 2
    assert b["append"] == 4 * 64 * 128 * 2


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mha", "--steps", "4", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_step_bytes_paged_and_mla():
    """A paged step adds the 4-byte table entries of the live rows; an MLA
    step reads each latent row once for all heads plus the two
    up-projections."""
    sys.path.insert(0, ROOT)
    import bench
    from static_kv_cache_gb300 import synth
    lengths = [1024, 17, 4000]
    dense = bench.step_bytes(synth.WORKLOADS["llama3_8b"].with_(batch=3), lengths)
    paged = bench.step_bytes(synth.WORKLOADS["llama3_8b_paged"].with_(batch=3), lengths)
    assert paged["attn"] - dense["attn"] == 4 * (64 + 2 + 250)
    assert paged["append"] == dense["append"]
    w = synth.WORKLOADS["mla_dsv2"].with_(batch=3)
    m = bench.step_bytes(w, lengths)
    assert m["attn"] == sum(lengths) * 512 * 2 + 2 * 3 * 16 * 128 * 2 + 2 * 16 * 128 * 512 * 2
    assert m["append"] == 2 * 3 * 512 * 2


def test_block_table_covers_the_live_rows_once():
    """The bench's paged inputs: each sequence gets ceil(valid / 16) distinct
    physical blocks of a pool of exactly that many, unused entries 0."""
    import numpy as np
    from static_kv_cache_gb300 import synth
    lengths = [1, 16, 17, 4096, 33]
    table, nb = synth.block_table(lengths, 4096, seed=3)
    need = [(n + 15) // 16 for n in lengths]
    assert nb == sum(need) and table.shape == (5, 256) and table.dtype == np.int32
    used = np.concatenate([table[b, :n] for b, n in enumerate(need)])
    assert sorted(used.tolist()) == list(range(nb))
    for b, n in enumerate(need):
        assert (table[b, n:] == 0).all()


def test_reference_arm_paged_and_mla_lines():
    """The reference arm runs the oracle's paged gather and its MLA decode
    on the same workloads the GPU arm measures."""
    for wl in ("llama3_8b_paged", "mla_dsv2"):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--workload", wl, "--steps", "2", "--warmup", "0"],
                           capture_output=True, text=True, timeout=600, cwd=ROOT)
        assert r.returncode == 0, r.stderr
        d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
        assert d["impl"] == "reference" and d["value"] > 0
        assert ("block table" in d["cpu_baseline"]["sample"]) == (wl == "llama3_8b_paged")
        assert ("MLA" in d["cpu_baseline"]["sample"]) == (wl == "mla_dsv2")
