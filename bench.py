#!/usr/bin/env python
"""Decode-step benchmark: append + decode attention over a static KV cache.

One step is the whole hot path for every layer of the workload: for each
layer, kvc_decode_step appends the new token's K/V rows at valid - 1 and
attends with one query row per head over the valid rows (one fused launch on
the tensor-core kernel, the append and the attention back to back
otherwise).  Every timed
step recomputes the same decode step (same positions), so all steps move the
same bytes.  Default workload: the Llama-3-8B-shaped GQA cache (32 layers,
B=16, H=32, H_kv=8, d_h=128, max_context 8192, bf16, ragged live lengths
uniform in [1024, 8192]).

Output: one JSON line on rank 0.  ``value`` is the algorithmic HBM traffic
of the step (K+V of the live rows + q + out for attention; k_new/v_new read
and written once for the append) per second of step time, summed over ranks.

``--impl reference`` times the fp64 CPU oracle instead (host cores only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from static_kv_cache_gb300 import synth  # noqa: E402

METRIC = "decode-attention HBM GB/s and % of GB300 peak; decode tokens/s per layer"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("static_kv_cache_gb300/csrc/kvc_decode.cuh",
                  "static_kv_cache_gb300/csrc/kvc_decode_mma.cuh",
                  "static_kv_cache_gb300/csrc/kvc_decode_tc.cuh",
                  "static_kv_cache_gb300/csrc/kvc_decode_q8.cuh",
                  "static_kv_cache_gb300/csrc/kvc_mla.cuh",
                  "static_kv_cache_gb300/csrc/kvc_internal.cuh",
                  "static_kv_cache_gb300/csrc/kvc_decode_inst.cu",
                  "static_kv_cache_gb300/csrc/kvc_api.cu")   # tensor-map boxes


def decode_kernel_name(w: synth.Workload) -> str:
    """The decode kernel the library picks for a workload: the tcgen05 kernel
    for contiguous 16-bit caches with 16- or 32-head groups at d_h 128, the
    mma.sync tensor-core kernel for 16-bit caches with head groups of 2 to 8,
    16, 32 or 64 and d_h of 64 or 128, the CUDA-core kernel otherwise."""
    if w.d_latent:
        return "mla_decode_kernel"
    if w.dtype == "int8":
        return "decode_q8_kernel"
    if w.dtype in ("bf16", "fp16") and w.group in (16, 32) and w.d_head == 128 and not w.paged:
        return "decode_tc_kernel"
    if w.dtype in ("bf16", "fp16") and (2 <= w.group <= 8 or w.group in (16, 32, 64)) and w.d_head in (64, 128):
        return "decode_mma_kernel"
    return "decode_split_kernel"


# --------------------------------------------------------------------------- helpers
def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=600)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("kvc", "reference"), default="kvc")
    p.add_argument("--workload", default="llama3_8b", choices=sorted(synth.WORKLOADS))
    p.add_argument("--layers", type=int, default=0,
                   help="use only this many layers of the workload (profiling small cases)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="wall time budget of the CPU-oracle baseline sample")
    p.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="time direct calls instead of a CUDA graph of one step")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="time only the headline workload (skip the other target configs)")
    return p.parse_args(argv)


# The other configurations the throughput target names (the Llama-2-70B layer
# at 32k, B=1 and B=4), the Qwen2.5 shape in both cache types and the 32-head
# multi-query shape: timed after the headline in the default single-GPU run
# and reported under "configs".
EXTRA_WORKLOADS = ("llama2_70b_b1", "llama2_70b_b4", "qwen2_5_1_5b_bf16", "qwen2_5_1_5b_fp32", "mqa_32h")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a scalar over all ranks (the slowest rank sets the job time)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step_per_rank: float, world: int, max_seconds: float, steps: int) -> float:
    """Whole-job GB/s: every rank moves the same bytes each step (weak
    scaling); the job takes as long as its slowest rank."""
    return bytes_per_step_per_rank * world * steps / max_seconds / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel from a committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    entry = d.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            sel = str(device_index)
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200", "-i", sel]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- workload
def step_bytes(w: synth.Workload, lengths) -> dict:
    """Algorithmic bytes of one layer's decode step (per launch).  An int8
    cache adds its 4-byte row scales to the rows read and written; its q,
    out and new rows are bf16.  A paged cache adds the 4-byte block-table
    entries of the live rows.  An MLA cache reads each latent row once for all
    heads, plus the two up-projections of the layer."""
    eb = synth.ELEM_BYTES[w.dtype]
    ab = synth.ELEM_BYTES[synth.ACT_DTYPE[w.dtype]]
    if w.d_latent:   # MLA: the latent rows once, q and out, both up-projections, the step's latent row
        live = int(np.asarray(lengths, dtype=np.int64).sum())
        attn = (live * w.d_latent * eb + 2 * w.batch * w.n_heads * w.d_head * ab
                + 2 * w.n_heads * w.d_head * w.d_latent * eb)
        return {"attn": attn, "append": 2 * w.batch * w.d_latent * eb}
    sb = 4 if w.dtype == "int8" else 0                          # scale bytes per cache row
    live = int(np.asarray(lengths, dtype=np.int64).sum())
    attn = 2 * w.n_kv_heads * (w.d_head * eb + sb) * live + 2 * w.batch * w.n_heads * w.d_head * ab
    append = 2 * w.batch * w.n_kv_heads * (w.d_head * ab + w.d_head * eb + sb)  # read k/v_new, write the rows
    if w.paged:   # the block table entries of the live rows, read once
        attn += 4 * int(((np.asarray(lengths, dtype=np.int64) + synth.BLOCK_ROWS - 1) // synth.BLOCK_ROWS).sum())
    return {"attn": attn, "append": append}


class DeviceState:
    """Caches, workspace, handle and the per-layer step inputs on one GPU."""

    # per-step inputs (attribute, keyword of step())
    STEP_INPUTS = (("q", "q"), ("k_new", "k_new"), ("v_new", "v_new"), ("valid_len", "vl"))

    def __init__(self, w: synth.Workload, device: int):
        from static_kv_cache_gb300 import kvc
        self.kvc = kvc
        self.w = w
        self.lengths = synth.live_lengths(w)
        self.maxlen = int(self.lengths.max())
        act = synth.ACT_DTYPE[w.dtype]
        tdt, adt = synth.DTYPES[w.dtype], synth.DTYPES[act]
        dev = torch.device("cuda", device)
        shape = (w.n_layers, w.batch, w.n_kv_heads, w.max_context, w.d_head)
        self.table = None
        if w.paged:
            table, self.num_blocks = synth.block_table(self.lengths.numpy(), w.max_context,
                                                       synth.sub_seed(w.seed, "table"))
            self.table = torch.from_numpy(table).to(dev)
            shape = (w.n_layers, self.num_blocks, w.n_kv_heads, synth.BLOCK_ROWS, w.d_head)
        self.K = torch.empty(shape, dtype=tdt, device=dev)
        self.V = torch.empty(shape, dtype=tdt, device=dev)
        self.KS = self.VS = None
        pre = (self.lengths - 1).tolist()
        if w.paged:
            synth.poison_(self.K, w.dtype)
            synth.poison_(self.V, w.dtype)
            R = synth.BLOCK_ROWS
            for layer in range(w.n_layers):
                for b in range(w.batch):
                    n = pre[b]
                    if n == 0:
                        continue
                    nb = (n + R - 1) // R
                    idx = self.table[b, :nb].long()
                    for pool, tag in ((self.K, "pk"), (self.V, "pv")):
                        rows = torch.empty((w.n_kv_heads, nb * R, w.d_head), dtype=tdt, device=dev)
                        synth.poison_(rows, w.dtype)
                        rows[:, :n] = synth.normal((w.n_kv_heads, n, w.d_head), w.dtype,
                                                   synth.sub_seed(w.seed, tag, layer, b), dev)
                        pool[layer].index_copy_(0, idx, rows.view(w.n_kv_heads, nb, R, w.d_head).transpose(0, 1))
        elif w.dtype == "int8":
            # codes uniform on [-127, 127], scales positive: synthetic rows as the
            # quantising append would leave them; scales past the live rows NaN
            self.KS = torch.full(shape[:-1], float("nan"), dtype=torch.float32, device=dev)
            self.VS = torch.full(shape[:-1], float("nan"), dtype=torch.float32, device=dev)
            g = synth.generator(synth.sub_seed(w.seed, "codes"), device=dev)
            self.K.copy_(torch.randint(-127, 128, shape, generator=g, device=dev, dtype=torch.int8))
            self.V.copy_(torch.randint(-127, 128, shape, generator=g, device=dev, dtype=torch.int8))
            for layer in range(w.n_layers):
                for b in range(w.batch):
                    n = pre[b]
                    if n:
                        self.KS[layer, b, :, :n] = torch.rand((w.n_kv_heads, n), generator=g, device=dev) * 0.03 + 0.002
                        self.VS[layer, b, :, :n] = torch.rand((w.n_kv_heads, n), generator=g, device=dev) * 0.03 + 0.002
        else:
            synth.poison_(self.K, w.dtype)
            synth.poison_(self.V, w.dtype)
            for layer in range(w.n_layers):
                for b in range(w.batch):
                    n = pre[b]
                    if n:
                        shp = (w.n_kv_heads, n, w.d_head)
                        self.K[layer, b, :, :n] = synth.normal(shp, w.dtype, synth.sub_seed(w.seed, "pk", layer, b), dev)
                        self.V[layer, b, :, :n] = synth.normal(shp, w.dtype, synth.sub_seed(w.seed, "pv", layer, b), dev)
        L, B = w.n_layers, w.batch
        self.q = synth.normal((L, B, w.n_heads, w.d_head), act, synth.sub_seed(w.seed, "q"), dev)
        self.k_new = synth.normal((L, B, w.n_kv_heads, 1, w.d_head), act, synth.sub_seed(w.seed, "kn"), dev)
        self.v_new = synth.normal((L, B, w.n_kv_heads, 1, w.d_head), act, synth.sub_seed(w.seed, "vn"), dev)
        self.out = torch.empty((L, B, w.n_heads, w.d_head), dtype=adt, device=dev)
        self.valid_len = self.lengths.to(dev)
        # the step is one launch: every decode kernel appends as it streams
        self.launches_per_layer = 1
        self.cfg = kvc.make_config(L, B, w.n_heads, w.n_kv_heads, w.d_head, w.max_context, w.dtype)
        self.ws = torch.empty(kvc.kvc_workspace_bytes(self.cfg), dtype=torch.uint8, device=dev)
        if w.paged:
            st, self.h = kvc.kvc_alloc_paged(self.cfg, self.K, self.V, self.num_blocks, self.table, self.ws,
                                             self.ws.numel())
        elif w.dtype == "int8":
            st, self.h = kvc.kvc_alloc_scaled(self.cfg, self.K, self.V, self.KS, self.VS, self.ws, self.ws.numel())
        else:
            st, self.h = kvc.kvc_alloc(self.cfg, self.K, self.V, self.ws, self.ws.numel())
        kvc.check(st, "kvc_alloc")
        torch.cuda.synchronize(dev)

    def step(self, stream, events=None, q=None, k_new=None, v_new=None, vl=None, out=None) -> int:
        """One decode step over all layers (append the new rows at valid_len - 1,
        then attend), one kvc_decode_step call per layer; returns the number
        of kernel launches."""
        kvc, w = self.kvc, self.w
        q = self.q if q is None else q
        k_new = self.k_new if k_new is None else k_new
        v_new = self.v_new if v_new is None else v_new
        vl = self.valid_len if vl is None else vl
        out = self.out if out is None else out
        sp = stream.cuda_stream
        for layer in range(w.n_layers):
            if events is not None:
                events[layer][0].record(stream)
            st = kvc.kvc_decode_step(self.h, layer, q[layer], k_new[layer], v_new[layer], vl, self.maxlen,
                                     out[layer], sp)
            if st:
                raise kvc.KvcError(st, "kvc_decode_step")
            if events is not None:
                events[layer][1].record(stream)
        return self.launches_per_layer * w.n_layers

    def error(self, stream) -> int:
        return self.kvc.kvc_get_error(self.h, stream.cuda_stream)

    def close(self):
        self.kvc.kvc_free(self.h)


class MlaState:
    """The MLA latent cache [L, B, max_context, d_latent], per-layer
    up-projections [L, H, d_h, d_latent] (entries N(0, 1/d_latent), so the
    rebuilt rows have unit variance), workspace, handle and step inputs."""

    STEP_INPUTS = (("q", "q"), ("c_new", "c_new"), ("valid_len", "vl"))

    def __init__(self, w: synth.Workload, device: int):
        from static_kv_cache_gb300 import kvc
        self.kvc = kvc
        self.w = w
        self.lengths = synth.live_lengths(w)
        self.maxlen = int(self.lengths.max())
        tdt = synth.DTYPES[w.dtype]
        dev = torch.device("cuda", device)
        L, B, H = w.n_layers, w.batch, w.n_heads
        self.C = torch.empty((L, B, w.max_context, w.d_latent), dtype=tdt, device=dev)
        synth.poison_(self.C, w.dtype)
        pre = (self.lengths - 1).tolist()
        for layer in range(L):
            for b in range(B):
                if pre[b]:
                    self.C[layer, b, :pre[b]] = synth.normal((pre[b], w.d_latent), w.dtype,
                                                             synth.sub_seed(w.seed, "pc", layer, b), dev)
        shape_w = (L, H, w.d_head, w.d_latent)
        self.wk = (synth.normal(shape_w, "fp32", synth.sub_seed(w.seed, "wk"), dev) / w.d_latent ** 0.5).to(tdt)
        self.wv = (synth.normal(shape_w, "fp32", synth.sub_seed(w.seed, "wv"), dev) / w.d_latent ** 0.5).to(tdt)
        self.q = synth.normal((L, B, H, w.d_head), w.dtype, synth.sub_seed(w.seed, "q"), dev)
        self.c_new = synth.normal((L, B, w.d_latent), w.dtype, synth.sub_seed(w.seed, "cn"), dev)
        self.out = torch.empty((L, B, H, w.d_head), dtype=tdt, device=dev)
        self.valid_len = self.lengths.to(dev)
        self.launches_per_layer = 3   # absorb (+ append), attention over the latents, combine + up-projection
        self.cfg = kvc.make_mla_config(L, B, H, w.d_head, w.d_latent, w.max_context, w.dtype)
        self.ws = torch.zeros(kvc.kvc_mla_workspace_bytes(self.cfg), dtype=torch.uint8, device=dev)
        st, self.h = kvc.kvc_mla_alloc(self.cfg, self.C, self.ws, self.ws.numel())
        kvc.check(st, "kvc_mla_alloc")
        torch.cuda.synchronize(dev)

    def step(self, stream, events=None, q=None, c_new=None, vl=None, out=None) -> int:
        """One MLA decode step over all layers: kvc_mla_decode_step per layer
        (append the latent row at valid_len - 1, attend, up-project)."""
        kvc, w = self.kvc, self.w
        q = self.q if q is None else q
        c_new = self.c_new if c_new is None else c_new
        vl = self.valid_len if vl is None else vl
        out = self.out if out is None else out
        sp = stream.cuda_stream
        for layer in range(w.n_layers):
            if events is not None:
                events[layer][0].record(stream)
            st = kvc.kvc_mla_decode_step(self.h, layer, q[layer], c_new[layer], self.wk[layer], self.wv[layer], vl,
                                         self.maxlen, out[layer], sp)
            if st:
                raise kvc.KvcError(st, "kvc_mla_decode_step")
            if events is not None:
                events[layer][1].record(stream)
        return self.launches_per_layer * w.n_layers

    def error(self, stream) -> int:
        return self.kvc.kvc_mla_get_error(self.h, stream.cuda_stream)

    def close(self):
        self.kvc.kvc_mla_free(self.h)


# --------------------------------------------------------------------------- CPU oracle sample
def cpu_oracle_sample(w: synth.Workload, seconds: float, host=None):
    """Time the fp64 oracle on a bounded sample of the workload: each sample
    step is the decode attention of one sequence (cycling over the batch) of
    layer 0, all its query heads.  Returns (GB/s, samples, seconds, threads)."""
    import oracle
    lengths = synth.live_lengths(w).numpy()
    if host is None:
        host = cpu_host_inputs(w, lengths)
    done_bytes, spent, n = 0, 0.0, 0
    while spent < seconds or n == 0:
        b = n % w.batch
        t0 = time.perf_counter()
        oracle_one(w, host, b, lengths)
        spent += time.perf_counter() - t0
        done_bytes += sample_bytes(w, lengths, b)
        n += 1
    return done_bytes / spent / 1e9, n, spent, oracle.num_threads()


def oracle_one(w: synth.Workload, host, b: int, lengths):
    """The oracle's decode attention of sequence b (layer 0); a paged cache
    is first gathered through its block table; an MLA cache goes through the
    MLA oracle (keys and values rebuilt from the latents)."""
    import oracle
    n = lengths[b:b + 1]
    if w.d_latent:
        Ch, wk, wv, qh = host
        return oracle.mla_decode_attn(qh[b:b + 1], Ch[b:b + 1, :int(n[0])], wk, wv, n, w.dtype)
    Kh, Vh, qh, table = host
    if table is not None:
        K = oracle.paged.gather(Kh, table[b:b + 1], int(n[0]))
        V = oracle.paged.gather(Vh, table[b:b + 1], int(n[0]))
    else:
        K, V = Kh[b:b + 1], Vh[b:b + 1]
    return oracle.decode_attn(qh[b:b + 1], K, V, n, oracle_dtype(w))


def sample_bytes(w: synth.Workload, lengths, b: int) -> int:
    """Algorithmic bytes of one oracle sample (one sequence, all heads)."""
    ab = synth.ELEM_BYTES[synth.ACT_DTYPE[w.dtype]]
    n = int(lengths[b])
    if w.d_latent:
        return n * w.d_latent * synth.ELEM_BYTES[w.dtype] + 2 * w.n_heads * w.d_head * ab
    table = 4 * ((n + synth.BLOCK_ROWS - 1) // synth.BLOCK_ROWS) if w.paged else 0
    return 2 * w.n_kv_heads * cache_row_bytes(w) * n + 2 * w.n_heads * w.d_head * ab + table


def cpu_host_inputs(w: synth.Workload, lengths):
    """Layer-0 inputs drawn on the host (same distribution and shapes).  For
    an int8 cache: rows quantised by the oracle and handed to it
    dequantised (fp64), q widened to fp64."""
    maxlen = int(np.max(lengths))
    act = synth.ACT_DTYPE[w.dtype]
    if w.d_latent:
        Ch = synth.to_bits(synth.normal((w.batch, maxlen, w.d_latent), w.dtype, synth.sub_seed(w.seed, "cpu_c"))).copy()
        wsh = (w.n_heads, w.d_head, w.d_latent)
        wk = synth.to_bits((synth.normal(wsh, "fp32", synth.sub_seed(w.seed, "cpu_wk")) / w.d_latent ** 0.5)
                           .to(synth.DTYPES[w.dtype]))
        wv = synth.to_bits((synth.normal(wsh, "fp32", synth.sub_seed(w.seed, "cpu_wv")) / w.d_latent ** 0.5)
                           .to(synth.DTYPES[w.dtype]))
        qh = synth.to_bits(synth.normal((w.batch, w.n_heads, w.d_head), w.dtype, synth.sub_seed(w.seed, "cpu_q")))
        return Ch, wk, wv, qh
    shape = (w.batch, w.n_kv_heads, maxlen, w.d_head)
    Kh = synth.to_bits(synth.normal(shape, act, synth.sub_seed(w.seed, "cpu_k"))).copy()
    Vh = synth.to_bits(synth.normal(shape, act, synth.sub_seed(w.seed, "cpu_v"))).copy()
    qh = synth.to_bits(synth.normal((w.batch, w.n_heads, w.d_head), act, synth.sub_seed(w.seed, "cpu_q")))
    if w.dtype == "int8":
        import oracle
        Kh = oracle.dequantize_rows(*oracle.quantize_rows(Kh, act))
        Vh = oracle.dequantize_rows(*oracle.quantize_rows(Vh, act))
        qh = oracle.widen(qh, act)
    table = None
    if w.paged:   # the same rows scattered into 16-row blocks of a pool
        table, nb = synth.block_table(lengths, w.max_context, synth.sub_seed(w.seed, "cpu_table"))
        R = synth.BLOCK_ROWS
        pools = []
        for dense in (Kh, Vh):
            pool = np.zeros((nb, w.n_kv_heads, R, w.d_head), dtype=dense.dtype)
            for b in range(w.batch):
                n = int(lengths[b])
                for j in range((n + R - 1) // R):
                    m = min(R, n - j * R)
                    pool[table[b, j], :, :m] = dense[b, :, j * R:j * R + m]
            pools.append(pool)
        Kh, Vh = pools
    return Kh, Vh, qh, table


def oracle_what(w: synth.Workload) -> str:
    if w.d_latent:
        return "MLA decode attention (keys and values rebuilt from the latents)"
    return ("gather through the block table and " if w.paged else "") + "decode attention"


def oracle_dtype(w: synth.Workload) -> str:
    return "fp64" if w.dtype == "int8" else w.dtype


def cache_row_bytes(w: synth.Workload) -> int:
    """Bytes of one cache row as stored (codes plus the scale for int8)."""
    return w.d_head * synth.ELEM_BYTES[w.dtype] + (4 if w.dtype == "int8" else 0)


def workload_config(w: synth.Workload, lengths, world: int) -> dict:
    if w.d_latent:
        return {"workload": f"{w.name}: MLA latent cache, {w.n_layers} layers, B={w.batch}, H={w.n_heads}, "
                            f"d_h={w.d_head}, d_latent={w.d_latent}, max_context={w.max_context}, {w.dtype} cache",
                "n_layers": w.n_layers, "batch": w.batch, "n_heads": w.n_heads, "d_head": w.d_head,
                "d_latent": w.d_latent, "max_context": w.max_context, "cache_dtype": w.dtype,
                "live_rows": int(np.asarray(lengths).sum()),
                "valid_len": "ragged U{%d..%d}" % w.ragged if w.ragged else "uniform %d" % int(lengths[0]),
                "l2": "inputs larger than L2: each layer's live latents exceed the 129 MB L2 and the layers are cycled",
                "parallelism": f"replicas x{world} (independent batches, no collective on the data path)"}
    return {"workload": f"{w.name}: {w.n_layers} layers, B={w.batch}, H={w.n_heads}, "
                        f"H_kv={w.n_kv_heads}, d_h={w.d_head}, max_context={w.max_context}, "
                        f"{w.dtype} cache",
            "n_layers": w.n_layers, "batch": w.batch, "n_heads": w.n_heads, "n_kv_heads": w.n_kv_heads,
            "d_head": w.d_head, "max_context": w.max_context, "cache_dtype": w.dtype,
            "live_rows_per_kv_head": int(np.asarray(lengths).sum()),
            "valid_len": "ragged U{%d..%d}" % w.ragged if w.ragged else "uniform %d" % int(lengths[0]),
            "layout": ("paged: 16-row blocks at random places in a pool of exactly the blocks the live rows need, "
                       "one int32 block table [B, max_context/16]") if w.paged else "contiguous [L, B, H_kv, max_context, d_h]",
            "l2": "inputs larger than L2: each layer's live K/V exceeds the 129 MB L2 and the layers are cycled",
            "parallelism": f"replicas x{world} (independent batches, no collective on the data path)"}


# --------------------------------------------------------------------------- arms
def time_steps(state, w, steps, warmup, no_graph, world, local, clocks=True) -> dict:
    """Warm up, then time `steps` whole decode steps on one stream between
    barrier + synchronize, with CUDA events at the two ends of the timed
    region only (an event between two launches would keep the second from
    overlapping the first's drain).  The steps replay a CUDA graph of
    `per_graph` consecutive steps captured from the same C-ABI calls a direct
    step makes (they only enqueue kernels), so launch-bound workloads measure
    the GPU rather than the host loop."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            state.step(stream)
    torch.cuda.synchronize()
    graph, graph_note = None, "direct calls (--no-graph)"
    per_graph = max(d for d in range(1, 9) if steps % d == 0)
    if not no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                g.capture_begin()
                try:
                    for _ in range(per_graph):
                        state.step(stream)
                finally:
                    g.capture_end()
            with torch.cuda.stream(stream):
                for _ in range(max(3, warmup)):
                    g.replay()
            torch.cuda.synchronize()
            graph, graph_note = g, f"CUDA graph of {per_graph} steps (every layer's call), replayed"
        except Exception as exc:  # capture not available: time direct calls
            graph, graph_note = None, f"direct calls (graph capture failed: {str(exc)[:120]})"
    launches_per_step = state.launches_per_layer * w.n_layers
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if clocks else None
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    launches = 0
    with torch.cuda.stream(stream):
        t_start.record(stream)
        if graph is not None:
            for _ in range(steps // per_graph):
                graph.replay()
                launches += launches_per_step * per_graph
        else:
            for _ in range(steps):
                launches += state.step(stream)
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = sampler.stop() if sampler else None
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed_max = reduce_max(elapsed, world, device=torch.device("cuda", local))
    err = state.error(stream)
    if err:
        raise state.kvc.KvcError(err, "device error word after the timed region")
    del graph
    return {"elapsed": elapsed, "elapsed_max": elapsed_max, "launches": launches, "launch": graph_note,
            "clocks": clk, "stream": stream}


def time_extra_configs(args, world, local, peak) -> dict:
    """The other target configurations, one after another (each one's
    buffers freed before the next): per config its whole-job GB/s, step
    time, fraction of the HBM peak and the clocks seen while it ran."""
    out = {}
    for name in EXTRA_WORKLOADS:
        w = synth.WORKLOADS[name]
        state = DeviceState(w, local)
        per_layer = step_bytes(w, state.lengths.numpy())
        bytes_call = per_layer["attn"] + per_layer["append"]
        # about half a second of timed steps at the expected rate, within [20, --steps]
        est_step_s = bytes_call * w.n_layers / (0.8 * peak * 1e9)
        steps = int(min(max(20, round(0.5 / est_step_s)), max(20, args.steps)))
        steps -= steps % 8 if steps >= 8 else 0
        r = time_steps(state, w, steps, max(3, args.warmup), args.no_graph, world, local, not args.no_clocks)
        call_s = r["elapsed"] / (steps * w.n_layers)
        achieved = bytes_call / call_s / 1e9
        out[name] = {
            "value": round(job_throughput(bytes_call * w.n_layers, world, r["elapsed_max"], steps), 2),
            "unit": UNIT, "steps": steps, "ms_per_step": round(r["elapsed_max"] / steps * 1e3, 4),
            "frac": round(achieved / peak, 4), "achieved": round(achieved, 2),
            "bytes_attn": per_layer["attn"], "bytes_append": per_layer["append"],
            "mean_call_us": round(call_s * 1e6, 3), "kernel": decode_kernel_name(w),
            "launches_per_call": state.launches_per_layer, "launch": r["launch"], "clocks": r["clocks"],
            "workload": workload_config(w, state.lengths.numpy(), world)["workload"],
        }
        state.close()
        del state
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def bench_kvc(args, rank, world, local):
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(n_layers=args.layers)
    state = MlaState(w, local) if w.d_latent else DeviceState(w, local)
    lengths = state.lengths.numpy()
    per_layer = step_bytes(w, lengths)
    bytes_step = (per_layer["attn"] + per_layer["append"]) * w.n_layers
    r = time_steps(state, w, args.steps, args.warmup, args.no_graph, world, local, not args.no_clocks)
    stream, graph_note, clocks, launches = r["stream"], r["launch"], r["clocks"], r["launches"]
    elapsed, elapsed_max = r["elapsed"], r["elapsed_max"]
    launches_per_call = state.launches_per_layer

    # --- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        host = {name: pin(getattr(state, name)) for name, _ in state.STEP_INPUTS}
        devin = {name: torch.empty_like(getattr(state, name)) for name, _ in state.STEP_INPUTS}
        kw = {arg: devin[name] for name, arg in state.STEP_INPUTS}
        hout = torch.empty(state.out.shape, dtype=state.out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = hout.numel() * hout.element_size()
        e2e_steps = max(3, min(args.steps, 200))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(e2e_steps):
                for name, _ in state.STEP_INPUTS:
                    devin[name].copy_(host[name], non_blocking=True)
                state.step(stream, **kw)
                hout.copy_(state.out, non_blocking=True)
                stream.synchronize()
        e2e_s = reduce_max(time.perf_counter() - t0, world, device=torch.device("cuda", local))
        e2e = {"value": round(job_throughput(bytes_step, world, e2e_s, e2e_steps), 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4)}

    # --- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        gbs, n, spent, threads = cpu_oracle_sample(w, args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"fp64 oracle {oracle_what(w)} of layer 0, one sequence (all {w.n_heads} heads) "
                         f"per sample, cycling over the batch: {n} samples in {spent:.1f} s"}

    value = job_throughput(bytes_step, world, elapsed_max, args.steps)
    peak, peak_src = load_peaks()
    extra = None
    if world == 1 and not args.no_extra and args.workload == "llama3_8b" and not args.layers:
        state.close()
        del state
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        state = None
        extra = time_extra_configs(args, world, local, peak)
    # one kvc call per layer and step; its average duration over the timed
    # region (gaps between calls included)
    mean_decode_s = elapsed / (args.steps * w.n_layers)
    achieved = (per_layer["attn"] + per_layer["append"]) / mean_decode_s / 1e9
    traffic = recorded_traffic(args.workload)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_max / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w, lengths, world),
                           accumulate="fp32 (products, softmax and sums; one rounding to the cache type at the end)"),
            "tokens_per_s_per_layer": round(world * w.batch * w.n_layers / (elapsed_max / args.steps), 1),
            "decode_tokens_per_s": round(world * w.batch / (elapsed_max / args.steps), 1),
            "decode_attn_pct_of_peak": round(100 * achieved / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": decode_kernel_name(w), "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback 6.8 TB/s",
                         "bytes_per_launch": per_layer["attn"] + per_layer["append"],
                         "bytes_attn": per_layer["attn"], "bytes_append": per_layer["append"],
                         "mean_launch_us": round(mean_decode_s * 1e6, 3),
                         "launches_per_call": launches_per_call,
                         "timing": "timed region / (steps x layers): one kvc decode-step call per layer, gaps included",
                         "launch": graph_note},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        }
        if extra is not None:
            line["configs"] = extra
        print(json.dumps(line), flush=True)
    if state is not None:
        state.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_reference(args, rank, world, local):
    """The oracle, as it stands, on the host cores: rank 0 only."""
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    if w.chunk:
        return bench_reference_prefill(args, world, w)
    lengths = synth.live_lengths(w).numpy()
    host = cpu_host_inputs(w, lengths)
    for _ in range(args.warmup):
        cpu_oracle_sample(w, 0.0, host)
    import oracle
    total_bytes, total_s, samples = 0.0, 0.0, 0
    for s in range(args.steps):
        if total_s > 12 * args.cpu_seconds:   # keep the whole run to a few minutes
            break
        b = s % w.batch
        t0 = time.perf_counter()
        oracle_one(w, host, b, lengths)
        total_s += time.perf_counter() - t0
        total_bytes += sample_bytes(w, lengths, b)
        samples += 1
    value = total_bytes / total_s / 1e9
    sample = (f"fp64 oracle {oracle_what(w)} of layer 0, "
              f"one sequence (all {w.n_heads} heads) per step, "
              f"cycling over the batch; {samples} steps in {total_s:.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / samples * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(workload_config(w, lengths, world),
                                                accumulate="fp64 (the oracle: exact widening, fp64 throughout)"),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- chunked prefill
PREFILL_METRIC = "chunked-prefill attention TFLOP/s"


def prefill_work(w: synth.Workload, prefix) -> dict:
    """Per layer: attention FLOPs (QK^T and PV, 2 FLOPs per multiply-add) of
    the chunk's causal rows, and the algorithmic bytes (K/V rows up to the
    chunk's end read once per KV head, q read, out written, the chunk's K/V
    appended)."""
    T, eb = w.chunk, synth.ELEM_BYTES[w.dtype]
    rows = sum(T * int(c) + T * (T + 1) // 2 for c in prefix)      # (query, key) pairs per head
    flops = 4 * w.d_head * w.n_heads * rows
    kv = 2 * w.n_kv_heads * w.d_head * eb * sum(int(c) + T for c in prefix)
    qo = 2 * w.batch * w.n_heads * T * w.d_head * eb
    app = 4 * w.batch * w.n_kv_heads * T * w.d_head * eb
    return {"flops": flops, "bytes": kv + qo + app}


class PrefillState:
    """Caches with the workload's live prefixes, and per layer one chunk of
    T_new rows to append at the prefix end and attend with."""

    def __init__(self, w: synth.Workload, device: int):
        from static_kv_cache_gb300 import kvc
        self.kvc, self.w = kvc, w
        self.prefix = synth.live_lengths(w)
        tdt = synth.DTYPES[w.dtype]
        dev = torch.device("cuda", device)
        L, B, T = w.n_layers, w.batch, w.chunk
        shape = (L, B, w.n_kv_heads, w.max_context, w.d_head)
        self.K = torch.empty(shape, dtype=tdt, device=dev)
        self.V = torch.empty(shape, dtype=tdt, device=dev)
        synth.poison_(self.K, w.dtype)
        synth.poison_(self.V, w.dtype)
        for layer in range(L):
            for b in range(B):
                n = int(self.prefix[b])
                if n:
                    shp = (w.n_kv_heads, n, w.d_head)
                    self.K[layer, b, :, :n] = synth.normal(shp, w.dtype, synth.sub_seed(w.seed, "pk", layer, b), dev)
                    self.V[layer, b, :, :n] = synth.normal(shp, w.dtype, synth.sub_seed(w.seed, "pv", layer, b), dev)
        self.q = synth.normal((L, B, w.n_heads, T, w.d_head), w.dtype, synth.sub_seed(w.seed, "q"), dev)
        self.k_new = synth.normal((L, B, w.n_kv_heads, T, w.d_head), w.dtype, synth.sub_seed(w.seed, "kn"), dev)
        self.v_new = synth.normal((L, B, w.n_kv_heads, T, w.d_head), w.dtype, synth.sub_seed(w.seed, "vn"), dev)
        self.out = torch.empty((L, B, w.n_heads, T, w.d_head), dtype=tdt, device=dev)
        self.cache_index = self.prefix.to(dev)
        self.cfg = kvc.make_config(L, B, w.n_heads, w.n_kv_heads, w.d_head, w.max_context, w.dtype)
        self.ws = torch.empty(kvc.kvc_workspace_bytes(self.cfg), dtype=torch.uint8, device=dev)
        st, self.h = kvc.kvc_alloc(self.cfg, self.K, self.V, self.ws, self.ws.numel())
        kvc.check(st, "kvc_alloc")
        torch.cuda.synchronize(dev)

    def step(self, stream, events=None, q=None, k_new=None, v_new=None, ci=None, out=None) -> int:
        """The chunk of every layer: append at the prefix end, then the
        prefill attention; returns the number of kernel launches."""
        kvc, w = self.kvc, self.w
        q = self.q if q is None else q
        k_new = self.k_new if k_new is None else k_new
        v_new = self.v_new if v_new is None else v_new
        ci = self.cache_index if ci is None else ci
        out = self.out if out is None else out
        sp = stream.cuda_stream
        for layer in range(w.n_layers):
            kvc.check(kvc.kvc_append(self.h, layer, k_new[layer], v_new[layer], ci, w.chunk, sp), "kvc_append")
            if events is not None:
                events[layer][0].record(stream)
            kvc.check(kvc.kvc_prefill_attn(self.h, layer, q[layer], ci, w.chunk, out[layer], sp), "kvc_prefill_attn")
            if events is not None:
                events[layer][1].record(stream)
        return 2 * w.n_layers

    def error(self, stream) -> int:
        return self.kvc.kvc_get_error(self.h, stream.cuda_stream)

    def close(self):
        self.kvc.kvc_free(self.h)


def cpu_prefill_sample(w: synth.Workload, seconds: float):
    """Time the fp64 oracle on a bounded sample of the prefill workload: each
    sample is 8 chunk rows of one sequence of layer 0 (all heads, causal over
    that sequence's prefix and chunk), cycling over the sequences."""
    import oracle
    prefix = synth.live_lengths(w)
    T, rows_per_sample = w.chunk, 8
    host = []
    for b in range(w.batch):
        c = int(prefix[b])
        ctx = c + T
        K = synth.normal((1, w.n_kv_heads, ctx, w.d_head), w.dtype, synth.sub_seed(w.seed, "cpu-k", b))
        V = synth.normal((1, w.n_kv_heads, ctx, w.d_head), w.dtype, synth.sub_seed(w.seed, "cpu-v", b))
        q = synth.normal((1, w.n_heads, rows_per_sample, w.d_head), w.dtype, synth.sub_seed(w.seed, "cpu-q", b))
        host.append((c, synth.to_bits(q), synth.to_bits(K), synth.to_bits(V)))
    flops, n, t0 = 0, 0, time.perf_counter()
    while True:
        c, q, K, V = host[n % len(host)]
        t = T - rows_per_sample    # the last rows of the chunk: the most keys
        oracle.prefill_attn(q, K, V, [c + t], rows_per_sample, w.dtype)
        flops += 4 * w.d_head * w.n_heads * sum(c + t + i + 1 for i in range(rows_per_sample))
        n += 1
        spent = time.perf_counter() - t0
        if spent >= seconds:
            break
    return flops / spent / 1e12, n, spent, oracle.num_threads()


def bench_prefill(args, rank, world, local):
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(n_layers=args.layers)
    state = PrefillState(w, local)
    work = prefill_work(w, state.prefix.numpy())
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            state.step(stream)
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in range(w.n_layers)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = None if args.no_clocks else ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    launches = 0
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for s_ in range(args.steps):
            launches += state.step(stream, evs[s_])
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    elapsed = reduce_max(t_start.elapsed_time(t_end) / 1e3, world, device=torch.device("cuda", local))
    launch_ms = [evs[s_][l][0].elapsed_time(evs[s_][l][1]) for s_ in range(args.steps) for l in range(w.n_layers)]
    err = state.error(stream)
    if err:
        raise state.kvc.KvcError(err, "device error word after the timed region")
    step_flops = work["flops"] * w.n_layers
    value = world * step_flops * args.steps / elapsed / 1e12

    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        hq, hk, hv, hci = pin(state.q), pin(state.k_new), pin(state.v_new), pin(state.cache_index)
        hout = torch.empty(state.out.shape, dtype=state.out.dtype).pin_memory()
        dq, dk, dv, dci = (torch.empty_like(x) for x in (state.q, state.k_new, state.v_new, state.cache_index))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hci))
        d2h = hout.numel() * hout.element_size()
        e2e_steps = max(3, min(args.steps, 50))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(e2e_steps):
                for d, hsrc in ((dq, hq), (dk, hk), (dv, hv), (dci, hci)):
                    d.copy_(hsrc, non_blocking=True)
                state.step(stream, q=dq, k_new=dk, v_new=dv, ci=dci)
                hout.copy_(state.out, non_blocking=True)
                stream.synchronize()
        e2e_s = reduce_max(time.perf_counter() - t0, world, device=torch.device("cuda", local))
        e2e = {"value": round(world * step_flops * e2e_steps / e2e_s / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_s / e2e_steps * 1e3, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        tf, n, spent, threads = cpu_prefill_sample(w, args.cpu_seconds)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"fp64 oracle prefill attention of layer 0, the last 8 chunk rows of one sequence "
                         f"(all {w.n_heads} heads) per sample, cycling over the batch: {n} samples in {spent:.1f} s"}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        peak, peak_src = float(pk["bf16_tflops_sustained"]), "measured (MEASURED_PEAKS.json bf16_tflops_sustained)"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 1700.0, "fallback 1.7 PFLOP/s sustained bf16"
    mean_launch_s = float(np.mean(launch_ms)) / 1e3
    achieved = work["flops"] / mean_launch_s / 1e12
    if rank == 0:
        line = {
            "metric": PREFILL_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{w.name}: {w.n_layers} layers, B={w.batch}, H={w.n_heads}, H_kv={w.n_kv_heads}, "
                                   f"d_h={w.d_head}, chunk T_new={w.chunk} after live prefixes U{w.ragged}, {w.dtype} cache",
                       "prefix_rows": [int(x) for x in state.prefix], "chunk": w.chunk,
                       "parallelism": f"replicas x{world}"},
            "prefill_tokens_per_s": round(world * w.batch * w.chunk / (elapsed / args.steps), 1),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": None, "kernel": "prefill_tc_kernel",
                         "peak_source": peak_src, "flops_per_launch": work["flops"],
                         "bytes_per_launch": work["bytes"],
                         "mean_launch_us": round(mean_launch_s * 1e6, 3)},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    state.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_reference_prefill(args, world, w):
    """The oracle's prefill attention on the host cores: each step one
    bounded sample (see cpu_prefill_sample) of about a second."""
    import oracle
    for _ in range(args.warmup):
        cpu_prefill_sample(w, 0.0)
    total_flops, total_s, samples = 0.0, 0.0, 0
    for _ in range(args.steps):
        tf, n, spent, _ = cpu_prefill_sample(w, 1.0)
        total_flops += tf * 1e12 * spent
        total_s += spent
        samples += n
    value = total_flops / total_s / 1e12
    sample = (f"fp64 oracle prefill attention of layer 0, the last 8 chunk rows of one sequence "
              f"(all {w.n_heads} heads) per sample, cycling over the batch; {samples} samples in {total_s:.1f} s")
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "chunk": w.chunk},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        bench_reference(args, rank, world, local)
    elif synth.WORKLOADS[args.workload].chunk:
        bench_prefill(args, rank, world, local)
    else:
        bench_kvc(args, rank, world, local)


if __name__ == "__main__":
    main()
