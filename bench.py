"""Benchmark: one paged-attention decode step (slot mapping -> KV write ->
decode attention) on the LLaMA-2-7B-shaped workload: B=64 sequences, context
lengths uniform in [512, 4096], 32 q heads = 32 kv heads, head_dim 128, fp16,
16-token blocks scattered over a pool 10% larger than needed.

Prints one JSON line.  After the headline (single GPU), every other workload
is timed for about a second on its own and summarised under "configs":
attention ms per launch, its roofline (HBM, or the tensor pipe for a call of
prefill chunks only) and the median SM clock of its timed region.
``--impl reference`` times the fp64 CPU oracle on the host cores instead (the
only baseline that exists for this path).
N > 1 (torchrun) runs independent replicas, one per GPU: the path has no
exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn decode tokens/s & HBM GB/s (% of GB300 peak), B=64 ctx≤4K"
UNIT = "tokens/s"
SPEC_HBM_GBS = 8000.0


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak(sustained: bool = False):
    """Dense bf16 tensor peak (TFLOP/s): the measured burst figure (a cuBLAS
    GEMM timed alone), or with `sustained` the figure of GEMMs run back to back
    for seconds under the power cap; else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def replica_throughput(world_size: int, units_per_step: int, steps: int, slowest_ms: float) -> float:
    """Units processed by all replicas per second, timed by the slowest rank."""
    return world_size * units_per_step * steps / (slowest_ms / 1e3)


def _algorithmic_bytes(w) -> dict:
    """Bytes the attention launch must move: every live K/V row once per kv
    head (a block shared by several sequences counts once: `kv_unique`; once
    per sequence that reads it: `kv`), the query rows, the output rows, the
    live table entries and the lengths."""
    n = w.seq_lens.astype(np.int64)
    row = w.num_kv_heads * w.head_dim * 2 * w.cache_elem_bytes   # K and V bytes of one token
    kv = int(n.sum()) * row
    rows_per_block = {}
    for b in range(w.batch):
        nb = -(-int(n[b]) // 16)
        for j in range(nb):
            blk = int(w.block_tables[b, j])
            rows_per_block[blk] = max(rows_per_block.get(blk, 0), min(16, int(n[b]) - 16 * j))
    kv_unique = sum(rows_per_block.values()) * row
    q = w.num_tokens * w.num_q_heads * w.head_dim * 2
    live_entries = int((-(-n // 16)).sum())
    meta = live_entries * 4 + w.batch * 4 * (1 if w.is_decode else 2)
    return {"kv": kv, "kv_unique": kv_unique, "q": q, "out": q, "meta": meta,
            "total": kv_unique + 2 * q + meta, "total_logical": kv + 2 * q + meta}


def _prefill_flops(w) -> float:
    """Dense-contraction FLOPs of the chunked-prefill rows: for a chunk of C
    new tokens on P cached ones, Hq * 4 * D * (C * P + C * (C + 1) / 2)."""
    f = 0.0
    for n, c in zip(w.seq_lens.astype(np.float64), w.q_lens.astype(np.float64)):
        if c > 1:
            p = n - c
            f += w.num_q_heads * 4.0 * w.head_dim * (c * p + c * (c + 1) / 2)
    return f


def _source_hash() -> str:
    """Hash of the decode kernel's source with comments and blank space
    removed, so that an edit to comments alone keeps a traffic record valid."""
    h = hashlib.sha256()
    for f in ("pa_decode.cu", "pa_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_attention_decode_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", "", text)                  # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def _traffic_per_launch(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_hash") != _source_hash() or d.get("workload") != workload:
            return None
        return int(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of the SM clock and the throttle
    reasons; `stop` summarises all of them, `window` those taken between two
    host times (time.time()) of the run."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.rows = []

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _when(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def _read(self):
        self.rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    self.rows.append(parts)
        os.unlink(self.path)

    @classmethod
    def summarise(cls, rows) -> dict | None:
        if not rows:
            return None
        try:
            sm = [float(r[2]) for r in rows]
            mx = max(float(r[3]) for r in rows)
        except ValueError:
            return None
        reasons = set()
        for r in rows:
            for name, val in zip(cls.REASONS, r[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(rows)}

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._read()
        return self.summarise(self.rows)

    def window(self, t0: float, t1: float) -> dict | None:
        """Summary of the samples taken between host times t0 and t1 (after stop)."""
        inside = [r for r in self.rows if (lambda t: t is not None and t0 <= t <= t1)(self._when(r[0]))]
        return self.summarise(inside)


def cpu_baseline(w, seconds: float = 10.0) -> dict:
    """Time the fp64 oracle (as it stands) on the host cores over whole
    sequences of the same workload: slot mapping, KV write and decode
    attention of each sampled sequence, cycling through the batch until about
    `seconds` of CPU time have been spent."""
    import oracle
    import torch

    def u16(t):
        return t.cpu().view(torch.int16).numpy().view(np.uint16)

    snaps = []
    for b in np.random.default_rng(7).permutation(w.batch)[: min(w.batch, 64)]:
        b = int(b)
        nb = -(-int(w.seq_lens[b]) // 16)
        idx = torch.from_numpy(w.block_tables[b, :nb].astype(np.int64)).to(w.k_cache.device)
        snaps.append((b, nb, u16(w.k_cache.index_select(0, idx)), u16(w.v_cache.index_select(0, idx)),
                      u16(w.q[b:b + 1]), u16(w.key[b:b + 1]), u16(w.value[b:b + 1])))
    done = tokens = 0
    t_total = 0.0
    while t_total < seconds or done == 0:
        b, nb, kc, vc, q, key, val = snaps[done % len(snaps)]
        tables = np.arange(nb, dtype=np.int32)[None, :]
        sl = w.seq_lens[b:b + 1]
        t0 = time.perf_counter()
        slots = oracle.slot_mapping(tables, sl, np.ones(1, np.int32), 16, nb)
        oracle.kv_write(key, val, kc, vc, slots)
        oracle.paged_attention_decode(q, kc, vc, tables, sl, w.scale, w.dtype)
        t_total += time.perf_counter() - t0
        done += 1
        tokens += int(sl[0])
    return {"value": done / t_total, "unit": UNIT, "cores": oracle.num_threads(0), "kind": "oracle",
            "sample": f"{done} whole sequences drawn from the workload ({len(snaps)} distinct, all "
                      f"{w.num_q_heads} heads, {tokens / done:.0f} context tokens on average): slot mapping "
                      f"+ KV write + decode attention in fp64, {t_total:.1f} s of CPU time"}


def _workload_kw(args) -> dict:
    if not args.batch:
        return {}
    if args.workload in ("mixed", "mixed_fp8"):
        return {"n_decode": args.batch}
    if args.workload in ("prefill", "prefill_fp8"):
        return {"n_prefill": args.batch}
    return {"batch": args.batch}


def _ctx(workload: str, w) -> str:
    """The context-length description of a workload for the JSON line."""
    if workload == "llama7b_decode":
        return f"U[512,4096] (mean {int(w.seq_lens.mean())})"
    return f"mean {int(w.seq_lens.mean())}, max {w.max_seq_len}"


def run_reference(args):
    """--impl reference: the oracle on the host cores, one whole sequence per step."""
    import oracle

    ws, rank, _ = _dist()
    if ws > 1 and rank != 0:
        return 0
    from paged_kv_attention_decode_gb300 import workloads as W

    import torch

    w = W.make(args.workload, device="cpu", **_workload_kw(args))
    if not w.is_decode:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times decode workloads only"}))
        return 0
    bt = w.block_tables

    def u16(t):
        return t.view(torch.int16).numpy().view(np.uint16)

    kcb, vcb, qb, keyb, valb = (u16(t) for t in (w.k_cache, w.v_cache, w.q, w.key, w.value))

    def step(i):
        b = i % w.batch
        sl = w.seq_lens[b:b + 1]
        tables = bt[b:b + 1]
        slots = oracle.slot_mapping(tables, sl, np.ones(1, np.int32), 16, w.num_blocks)
        oracle.kv_write(keyb[b:b + 1], valb[b:b + 1], kcb, vcb, slots)
        oracle.paged_attention_decode(qb[b:b + 1], kcb, vcb, tables, sl, w.scale, w.dtype)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": w.batch, "ctx": _ctx(args.workload, w),
                   "heads": f"{w.num_q_heads}/{w.num_kv_heads}", "head_dim": w.head_dim, "block_size": 16,
                   "step": "one whole sequence per step (rotating through the batch)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(0), "kind": "oracle",
                         "sample": "one whole sequence of the workload per step: slot mapping + KV write "
                                   "+ decode attention, fp64"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _compact(x):
    """Floats of the JSON line to 6 significant digits (the line stays short
    enough for a log tail to carry it whole)."""
    if isinstance(x, float):
        return float(f"{x:.6g}")
    if isinstance(x, dict):
        return {k: _compact(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [_compact(v) for v in x]
    return x


# Workloads timed after the headline, one at a time (each freed before the
# next), each for about SWEEP_SECONDS: every other configuration's attention
# call with its roofline and the SM clock seen during its own timed region.
SWEEP = ("llama7b_ctx4096", "gqa_prefix", "long_context", "mixed", "llama7b_decode_fp8", "mixed_fp8", "prefill",
         "prefill_fp8", "spec_verify")
SWEEP_SECONDS = 1.0


class Run:
    """One workload resident on the device and its step: slot mapping + KV
    write (`write`), then the attention call (`attend`), all through the
    library's public Python API."""

    def __init__(self, pa, W, name: str, dev, partition: int, kw: dict):
        import torch

        self.pa = pa
        self.name = name
        w = self.w = W.make(name, device=dev, **kw)
        self.T = w.num_tokens
        self.decode = w.is_decode
        self.fp8 = w.meta.get("cache_dtype") == "fp8"
        self.kv_scale = w.meta.get("kv_scale", 1.0)
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.sl = torch.from_numpy(w.seq_lens).to(dev)
        self.cu = None if self.decode else torch.from_numpy(w.cu_q_lens).to(dev)
        self.slots = torch.empty(self.T, dtype=torch.int64, device=dev)
        self.out = torch.empty_like(w.q)
        self.partition_arg = partition if self.decode else 0
        # FP8 chunks longer than 8 queries: the 16-bit copy of their blocks
        # (sized from the workload's host arrays, as a scheduler would)
        self.chunk_kv = int(w.seq_lens[w.q_lens > 8].astype(np.int64).sum()) if self.fp8 and not self.decode else 0
        if self.decode:
            nbytes = pa.decode_workspace_bytes(w.batch, w.num_q_heads, w.head_dim, w.max_seq_len, partition)
        elif self.fp8 and w.max_q_len > 8:
            nbytes = pa.prefill_fp8_workspace_bytes(w.batch, self.T, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                    w.max_seq_len, w.max_blocks_per_seq, self.chunk_kv)
        else:
            nbytes = pa.prefill_workspace_bytes(w.batch, self.T, w.num_q_heads, w.head_dim, w.max_seq_len)
        self.wsp = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.max_len = w.max_seq_len
        self.partition = pa.decode_partition(self.max_len, self.partition_arg)
        parts = -(-self.max_len // self.partition)
        # slot mapping + KV write; the decode plan + decode kernels; the
        # log-sum-exp reduce when a sequence can span several partitions; the
        # prefill plan + prefill kernels when a chunk is longer than 8 queries
        # (and, over an FP8 cache, the kernel that widens the chunks' blocks)
        chunks = not self.decode and w.max_q_len > 8
        self.launches_per_step = 4 + (1 if parts > 1 else 0) + (2 if chunks else 0) + (1 if chunks and self.fp8 else 0)

    def write(self, key=None, value=None, bt=None, sl=None, cu=None):
        pa, w = self.pa, self.w
        pa.slot_mapping(self.bt if bt is None else bt, self.sl if sl is None else sl,
                        self.cu if cu is None else cu, self.T, w.num_blocks, out=self.slots)
        key = w.key if key is None else key
        value = w.value if value is None else value
        if self.fp8:
            pa.paged_kv_write_fp8(key, value, w.k_cache, w.v_cache, self.slots, self.kv_scale, self.kv_scale)
        else:
            pa.paged_kv_write(key, value, w.k_cache, w.v_cache, self.slots)

    def attend(self, q=None, bt=None, sl=None, cu=None):
        pa, w = self.pa, self.w
        q = w.q if q is None else q
        bt = self.bt if bt is None else bt
        sl = self.sl if sl is None else sl
        if self.fp8 and self.decode:
            pa.paged_attention_decode_fp8(q, w.k_cache, w.v_cache, bt, sl, w.scale, self.kv_scale, self.kv_scale,
                                          self.max_len, out=self.out, partition_size=self.partition_arg,
                                          workspace=self.wsp)
        elif self.fp8:
            pa.paged_attention_prefill_fp8(q, w.k_cache, w.v_cache, bt, sl, self.cu if cu is None else cu, w.scale,
                                           self.kv_scale, self.kv_scale, w.max_q_len, self.max_len, out=self.out,
                                           workspace=self.wsp, chunk_kv_tokens=self.chunk_kv)
        elif self.decode:
            pa.paged_attention_decode(q, w.k_cache, w.v_cache, bt, sl, w.scale, self.max_len, out=self.out,
                                      partition_size=self.partition_arg, workspace=self.wsp)
        else:
            pa.paged_attention_prefill(q, w.k_cache, w.v_cache, bt, sl, self.cu if cu is None else cu, w.scale,
                                       w.max_q_len, self.max_len, out=self.out, workspace=self.wsp)

    def step(self):
        self.write()
        self.attend()

    def timed(self, steps: int, stream):
        """CUDA events around each step's write and attention call, on the
        launch stream: (whole-run ms, mean attention ms, mean write ms)."""
        import torch

        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for e0, e1, e2 in ev:
            e0.record(stream)
            self.write()
            e1.record(stream)
            self.attend()
            e2.record(stream)
        torch.cuda.synchronize()
        total_ms = ev[0][0].elapsed_time(ev[-1][2])
        attn_ms = sum(e1.elapsed_time(e2) for _, e1, e2 in ev) / steps
        write_ms = sum(e0.elapsed_time(e1) for e0, e1, _ in ev) / steps
        return total_ms, attn_ms, write_ms

    def roofline(self, attn_ms: float) -> dict:
        """Roofline of the attention call: algorithmic bytes over HBM, or, for
        a call of chunked-prefill rows only, algorithmic FLOPs over the dense
        bf16 tensor peak."""
        w = self.w
        if not self.decode and int(w.q_lens.min()) > 8:
            tpeak, tkind = _tensor_peak()
            fl = _prefill_flops(w)
            tf = fl / (attn_ms / 1e3) / 1e12
            return {"bound": "tensor", "achieved": tf, "peak": tpeak, "unit": "TFLOP/s", "frac": tf / tpeak,
                    "peak_kind": f"{tkind} dense bf16 GEMM (burst)", "algorithmic_flops_per_launch": fl,
                    "frac_of_sustained": tf / _tensor_peak(sustained=True)[0]}
        peak, kind = _peaks()
        ab = _algorithmic_bytes(w)
        gbs = ab["total"] / (attn_ms / 1e3) / 1e9
        r = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
             "peak_kind": f"{kind} HBM copy", "frac_of_8TBs_spec": gbs / SPEC_HBM_GBS,
             "algorithmic_bytes_per_launch": ab["total"]}
        if ab["kv"] != ab["kv_unique"]:
            r["logical_gbs"] = ab["total_logical"] / (attn_ms / 1e3) / 1e9
        return r


def _sig(x: float, digits: int = 4):
    return float(f"{x:.{digits}g}")


def sweep(pa, W, dev, stream, partition: int, warmup: int, names=SWEEP, seconds: float = SWEEP_SECONDS) -> dict:
    """Time each named workload's step on its own for about `seconds`; one
    compact record per workload (attention ms per launch, its roofline and the
    median SM clock of its timed region)."""
    import torch

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.5)
    windows, rows = {}, {}
    for name in names:
        r = Run(pa, W, name, dev, partition, {})
        for _ in range(max(warmup, 3)):
            r.step()
        est_total, _, _ = r.timed(5, stream)
        steps = int(min(4000, max(20, seconds * 1e3 / max(est_total / 5, 1e-3))))
        t0 = time.time()
        total_ms, attn_ms, write_ms = r.timed(steps, stream)
        windows[name] = (t0, time.time())
        rl = r.roofline(attn_ms)
        # achieved is GB/s for an "hbm" bound, TFLOP/s for "tensor"
        rows[name] = {"ms": _sig(attn_ms), "write_ms": _sig(write_ms, 3), "steps": steps, "bound": rl["bound"],
                      "achieved": _sig(rl["achieved"]), "frac": _sig(rl["frac"], 3)}
        if "logical_gbs" in rl:
            rows[name]["logical"] = _sig(rl["logical_gbs"])
        if "frac_of_sustained" in rl:   # (the loop runs about a second: it may meet the power cap)
            rows[name]["frac_sust"] = _sig(rl["frac_of_sustained"], 3)
        del r
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    clocks.stop()
    for name, (t0, t1) in windows.items():
        c = clocks.window(t0, t1)
        rows[name]["sm_mhz"] = c["sm_mhz"] if c else None
        if c and c["reasons"]:
            rows[name]["reasons"] = c["reasons"]
    return rows


def run_ours(args):
    import torch

    import paged_kv_attention_decode_gb300 as pa
    from paged_kv_attention_decode_gb300 import workloads as W

    ws, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pa.load_library()
    stream = torch.cuda.current_stream()

    r = Run(pa, W, args.workload, dev, args.partition, _workload_kw(args))
    w, T, decode, fp8 = r.w, r.T, r.decode, r.fp8
    B = w.batch
    for _ in range(args.warmup):
        r.step()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.5)
    if dist:
        dist.barrier()
    total_ms, attn_ms, write_ms = r.timed(args.steps, stream)
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = max_over_ranks(total_ms, dist, dev)
    value = replica_throughput(ws, T, args.steps, total_ms)

    # ---- end to end through the public API with host buffers -------------
    # Every step copies its inputs from pinned host memory and its output
    # back.  Two input sets make a two-deep pipeline, as a serving loop would
    # run it: step i+1's inputs travel on a copy stream while step i computes.
    q_h = w.q.cpu().pin_memory()
    k_h = w.key.cpu().pin_memory()
    v_h = w.value.cpu().pin_memory()
    bt_h = torch.from_numpy(w.block_tables).pin_memory()
    sl_h = torch.from_numpy(w.seq_lens).pin_memory()
    cu_h = None if decode else torch.from_numpy(w.cu_q_lens).pin_memory()
    out_h = [torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory() for _ in range(2)]
    host_in = [t for t in (q_h, k_h, v_h, bt_h, sl_h, cu_h) if t is not None]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = out_h[0].numel() * out_h[0].element_size()
    sets = [[torch.empty(t.shape, dtype=t.dtype, device=dev) for t in host_in] for _ in range(2)]
    e2e_steps = max(10, min(args.steps, 500))
    copy_stream = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def stage(i):
        k = i % 2
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(comp_done[k])       # step i-2 is done with this set
            for d, h in zip(sets[k], host_in):
                d.copy_(h, non_blocking=True)
            h2d_done[k].record(copy_stream)

    def e2e_run(n):
        stage(0)
        for i in range(n):
            if i + 1 < n:
                stage(i + 1)
            k = i % 2
            stream.wait_event(h2d_done[k])
            q_d, k_d, v_d, bt_d, sl_d = sets[k][:5]
            cu_d = sets[k][5] if cu_h is not None else None
            r.write(k_d, v_d, bt_d, sl_d, cu_d)
            r.attend(q_d, bt_d, sl_d, cu_d)
            out_h[k].copy_(r.out, non_blocking=True)
            comp_done[k].record(stream)
        stream.synchronize()
        copy_stream.synchronize()

    e2e_run(3)
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, dist, dev)
    e2e_value = replica_throughput(ws, T, e2e_steps, e2e_s * 1e3)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    ab = _algorithmic_bytes(w)
    rl = r.roofline(attn_ms)
    rl["ms_per_launch"] = attn_ms
    if rl["bound"] == "hbm":
        rl["traffic"] = _traffic_per_launch(args.workload)
        rl["kernel"] = ("decode attention call (work-list plan + persistent decode kernel + log-sum-exp reduce)"
                        if decode or w.max_q_len <= 8 else
                        "attention call (decode and verify rows: plan + decode + reduce kernels; longer chunks: "
                        "prefill plan + tcgen05 prefill kernel)")
    else:
        rl["traffic"] = None
        rl["kernel"] = "prefill call (prefill plan + tcgen05 prefill kernel)"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 cache, " if fp8 else "") + ("f16" if w.dtype == "f16" else "bf16"),
        "data": "synthetic",
        "config": {"workload": args.workload, "batch": B, "new_tokens_per_step": T, "ctx": _ctx(args.workload, w),
                   "heads": f"{w.num_q_heads}/{w.num_kv_heads}", "head_dim": w.head_dim, "block_size": 16,
                   "partition": r.partition, "pool_blocks": w.num_blocks,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {ab['kv_unique'] / 1e9:.2f} GB of KV read per step"},
        "roofline": rl,
        "write_ms_per_step": write_ms,
        "attention_tokens_per_s": T / (attn_ms / 1e3),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "pipeline": "2-deep: next step's inputs copied on a second stream"},
        "gpu_launches": r.launches_per_step * args.steps,
        "clocks": clk,
    }
    if not decode:
        line["prefill_gflop_per_step"] = _prefill_flops(w) / 1e9
    if ws == 1 and decode and not fp8 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, seconds=args.cpu_seconds)
    del r, w, sets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if ws == 1 and not args.no_sweep:
        names = [n for n in ("llama7b_decode",) + SWEEP if n != args.workload]
        line["configs"] = sweep(pa, W, dev, stream, args.partition, 5, names)
    print(json.dumps(_compact(line)), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    from paged_kv_attention_decode_gb300.workloads import CONFIGS
    ap.add_argument("--workload", default="llama7b_decode", choices=sorted(CONFIGS),
                    help="synthetic workload (default: the B=64 LLaMA-2-7B-shaped decode step)")
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the short timing of the other workloads after the headline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
