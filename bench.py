"""Benchmark of KV-outer block-sparse paged attention (index + forward +
combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all]
                    [--impl reference]

One step is one pass of the whole path (sa_attention: CSR index build,
KV-outer forward, log-sum-exp combine) over one batch of the workload, with
every input resident in HBM.  Between timed steps L2 is flushed by writing a
512 MiB buffer (outside the step's CUDA events).  Prints one JSON line.

With --workload all (the default) the headline is the long-context decode
workload (128 sequences of one query over 64-131 K keys, a 69 GB bf16 K/V
pool: the largest single-GPU configuration) and the line carries one
sub-record per other serving workload (GQA decode, chunked prefill with f32
and with bf16 K/V, skewed selection), each measured the same way with its
own steps, roofline, end-to-end rate and CPU baseline.

The CPU baseline is the oracle (plain f64 C) as it stands, run on the host's
cores by one thread per core over a bounded sample of the workload: shards of
(sequence, kv head, query rows), each an independent sub-problem because a
q-head reads only its own kv head.  --impl reference times the same oracle,
every step one such sample.

Under torchrun (N > 1) every rank runs its own replica of the workloads (its
own seed) on its own GPU: the path has no exchange step, so there is no data
collective; a barrier and a max-reduction of the elapsed time bracket each
timed region.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn fwd queries/s + selected-KV GB/s (% of GB300 HBM roofline)"
UNIT = "queries/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
SPLIT_EDGES = {"tiny": 0, "gqa_decode": 0, "chunked_prefill": 16, "chunked_prefill_bf16": 16,
               "skewed": 16, "long_decode": 0}
HEADLINE = "long_decode"
SUB_WORKLOADS = ("gqa_decode", "chunked_prefill", "chunked_prefill_bf16", "skewed")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all",
                    help="'all' (headline long_decode + the other serving workloads as "
                         "sub-records) or one workload name")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=4.0,
                    help="wall seconds of oracle work per phase of each CPU baseline")
    ap.add_argument("--partials", default="f32", choices=["f32", "bf16"],
                    help="o partial storage: f32 (the pages' layout) or the opt-in bf16")
    return ap.parse_args()


def make_workload(name: str, seed: int):
    """The five serving workloads, plus reduced-pool variants used only for
    ncu captures (same per-unit work, pool of a few GB)."""
    import inputs

    if name == "gqa_decode_ncu":
        w = inputs.gqa_decode(seed, kv_min=4096, kv_max=6144)
        w.name = name
        return w
    if name == "chunked_prefill_ncu":
        w = inputs.chunked_prefill(seed, batch=1)
        w.name = name
        return w
    if name == "chunked_prefill_bf16_ncu":
        w = inputs.chunked_prefill(seed, batch=1, kv_dtype="bf16")
        w.name = name
        return w
    if name == "skewed_ncu":
        w = inputs.skewed(seed, batch=4)
        w.name = name
        return w
    if name == "long_decode_ncu":
        w = inputs.long_decode(seed, batch=128, kv_min=8192, kv_max=12288)
        w.name = name
        return w
    if name.endswith("_idx"):
        # captures of the index kernel: the full workload's selection, lengths
        # and tables (so the same index work), its block tables folded onto a
        # pool of 8192 pages so that the capture holds little device memory
        w = inputs.FULL[name[:-4]](seed)
        w.block_tables = np.where(w.block_tables >= 0, w.block_tables % 8192, -1).astype(np.int32)
        w.num_pages = 8192
        w.name = name
        return w
    return inputs.FULL[name](seed)


# --------------------------------------------------------------------------- accounting


def algorithmic_bytes(w, fused=False, o_bytes=4) -> dict:
    """Bytes the KV-outer method must move, from the workload's own index
    inputs: each kept (kv head, block) loads its live keys' K and V once, Q is
    read once, the partials are written by the forward and read by the
    combine (o at o_bytes per value: 4, or 2 for the opt-in bf16 o partials;
    m and l at 4), the output is written once.  On the fused decode path the
    partials stay on chip, so its one kernel ("forward") moves K, V, Q, the
    index's inv rows and the output."""
    elt = 2 if w.kv_dtype == "bf16" else 4
    cu = w.cu_seqlens_q
    kv_keys = 0
    flops = 0
    edges = 0
    for b in range(w.batch):
        q0, q1 = int(cu[b]), int(cu[b + 1])
        if q1 == q0:
            continue
        lk = max(int(w.used_kv_lens[b]), 0) if w.pass_used else w.msb * w.block_size
        sel = w.selected[q0:q1]                                   # [qo, hkv, topk]
        kept = (sel >= 0) & (sel.astype(np.int64) * w.block_size < lk)
        edges += int(kept.sum())
        live_pages = (w.block_tables[b] >= 0)
        for h in range(w.hkv):
            blocks = np.unique(sel[:, h][kept[:, h]])
            for blk in blocks:
                s0 = int(blk) * w.block_size
                s1 = min(s0 + w.block_size, lk)
                pos = np.arange(s0, s1)
                nk = int(np.sum(live_pages[pos // w.page_size]))
                kv_keys += nk
                n_e = int(np.sum(sel[:, h][kept[:, h]] == blk))
                flops += 4 * w.head_dim * nk * n_e * w.qhead        # upper bound (no causal cut)
    kv = 2 * kv_keys * w.head_dim * elt
    q = w.tq * w.hq * w.head_dim * 4
    parts = edges * w.qhead * (w.head_dim * o_bytes + 2 * 4)
    out = w.tq * w.hq * w.head_dim * 4
    inv = w.hkv * w.tq * w.topk * 4
    if fused:
        return {"kv": kv, "q": q, "partials_write": 0, "partials_read": 0, "out": out,
                "inv": inv, "edges": edges, "flops": flops,
                "forward": kv + q + out + inv, "combine": 0, "step": kv + q + out + inv}
    return {"kv": kv, "q": q, "partials_write": parts, "partials_read": parts, "out": out,
            "inv": inv, "edges": edges, "flops": flops,
            "forward": kv + q + parts, "combine": parts + inv + out,
            "step": kv + q + 2 * parts + out}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_digest(path: str) -> str:
    """sha256 (16 hex digits) of a CUDA source's code: comments, trailing
    blanks and empty lines removed, so that a comment edit does not detach a
    profile from the code it was taken on."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def ncu_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current code (else None)."""
    src = os.path.join(ROOT, "block_sparse_paged_csr_gb300", "csrc", kernel_file)
    prof = os.path.join(ROOT, "profiles", f"{kernel_file.split('.')[0]}_{workload}.md")
    if not (os.path.exists(src) and os.path.exists(prof)):
        return None
    text = open(prof).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(code sha256 ([0-9a-f]+)\)",
                  text)
    if not m or m.group(2) != code_digest(src):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        deadline = time.time() + 5
        while not self.lines and time.time() < deadline:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if self.t0 - 0.06 <= t <= self.t1 + 0.06] or \
            [l for (_, l) in self.lines[-3:]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- ours


def aggregate_ranks(elapsed_s, e2e_per_rank, world, device):
    """Whole-job figures of a replicated run: the slowest rank's elapsed time
    (every rank did the same amount of work) and the end-to-end throughput as
    world x the slowest rank's.  world = 1 returns the inputs unchanged."""
    if world <= 1:
        return elapsed_s, e2e_per_rank
    import torch
    import torch.distributed as dist

    t = torch.tensor([elapsed_s], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    elapsed = float(t.item())
    e2e_total = None
    if e2e_per_rank is not None:
        t = torch.tensor([e2e_per_rank], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MIN)
        e2e_total = float(t.item()) * world
    return elapsed, e2e_total


def job_throughput(queries_per_step, steps, world, elapsed_s):
    """Queries per second of the whole job: every rank ran `steps` steps of
    `queries_per_step` queries; the job took the slowest rank's time."""
    return world * queries_per_step * steps / elapsed_s


def measure_workload(name, args, rank, world, local_rank):
    """Time K steps of sa_attention on one workload (plus per-stage and
    end-to-end timings).  Returns (record or None on ranks > 0, workload)."""
    import torch

    import block_sparse_paged_csr_gb300 as sa
    import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = make_workload(name, args.seed + rank)
    split = SPLIT_EDGES.get(name.replace("_ncu", ""), 0)
    fwd_kernel = sa.sa_attention_kernel_name(w.cu_seqlens_q, w.num_pages, w.hkv, w.hq,
                                             w.head_dim, w.block_size, w.page_size, w.kv_dtype,
                                             causal=w.causal)
    fused = fwd_kernel == "fused_dec_kernel"
    acct = algorithmic_bytes(w, fused, o_bytes=2 if args.partials == "bf16" else 4)

    q, k, v = inputs.device_tensors(w, dev)
    sel = torch.from_numpy(w.selected).to(dev)
    cu = torch.from_numpy(w.cu_seqlens_q).to(dev)
    used = torch.from_numpy(w.used_kv_lens).to(dev) if w.pass_used else None
    bt = torch.from_numpy(w.block_tables).to(dev)
    cu_host = w.cu_seqlens_q
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(index=None, partials=None, out=None, lse=None):
        return sa.sa_attention(q, k, v, sel, cu_host, cu, used, bt, w.hq, w.hkv, w.head_dim,
                               w.block_size, w.page_size, w.softmax_scale, w.causal,
                               split_edges=split, index=index, partials=partials, out=out,
                               lse=lse, partial_dtype=args.partials if partials is None else None)

    out, lse, index, partials = step()
    torch.cuda.synchronize(dev)
    status = sa.sa_get_status(index)
    if status != 0:
        raise RuntimeError(f"{name}: device status {sa.sa_status_string(status)}")
    for _ in range(max(args.warmup, 3)):
        step(index, partials, out, lse)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- timed region: K steps of the whole path -----------------------------
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    clocks.mark(True)
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush.fill_(float(s))
        starts[s].record(stream)
        step(index, partials, out, lse)
        ends[s].record(stream)
    barrier()
    wall = time.perf_counter() - t_wall
    clocks.mark(False)
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = float(sum(step_ms))
    status = sa.sa_get_status(index)
    if status != 0:
        raise RuntimeError(f"{name}: device status {sa.sa_status_string(status)}")

    # ---- per-stage durations (same launches, events between the stages) -----
    # On the fused decode path steps 2 and 3 are one kernel (sa_forward_combine).
    n_stage = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_stage)]
    o_p, m_p, l_p = partials
    for s in range(n_stage):
        flush.fill_(float(s))
        e = ev[s]
        e[0].record(stream)
        sa.sa_build_index(sel, cu_host, cu, used, w.max_pages, w.block_size, w.page_size,
                          split_edges=split, index=index)
        e[1].record(stream)
        if fused:
            sa.sa_forward_combine(q, k, v, index, sel, cu_host, cu, used, bt, w.hq, w.head_dim,
                                  w.block_size, w.page_size, w.softmax_scale, w.causal,
                                  split_edges=split, partials=partials, out=out, lse=lse)
            e[2].record(stream)
        else:
            # as inside sa_attention: the tensor-core forward keeps a bf16
            # copy of Q in `out` (written only by the combine)
            sa.sa_forward(q, k, v, index, bt, cu, used, w.hq, w.hkv, w.head_dim, w.block_size,
                          w.page_size, w.softmax_scale, w.causal, o_p, m_p, l_p, q_scratch=out)
            e[2].record(stream)
            sa.sa_combine(index, o_p, m_p, l_p, w.hq, w.head_dim, out, lse)
        e[3].record(stream)
    torch.cuda.synchronize(dev)
    st = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev])
    index_ms, fwd_ms, comb_ms = (float(x) for x in st.mean(axis=0))

    # f32 K/V on the tensor-core kernel: bf16 operands by default; the
    # opt-in tf32 scores are timed beside them (forward stage only)
    tf32_scores = None
    if fwd_kernel == "forward_tc_kernel" and w.kv_dtype == "f32":
        eb = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_stage)]
        for s_ in range(n_stage):
            flush.fill_(float(s_))
            eb[s_][0].record(stream)
            sa.sa_forward(q, k, v, index, bt, cu, used, w.hq, w.hkv, w.head_dim, w.block_size,
                          w.page_size, w.softmax_scale, w.causal, o_p, m_p, l_p, q_scratch=out,
                          path=sa.PATH_TENSOR_CORE_TF32)
            eb[s_][1].record(stream)
        torch.cuda.synchronize(dev)
        bms = float(np.mean([x[0].elapsed_time(x[1]) for x in eb]))
        tf32_scores = {"forward_ms": bms,
                       "roofline_frac": acct["forward"] / (bms / 1e3) / 1e9 / measured_peak()[0],
                       "note": "sa_forward with SA_PATH_TENSOR_CORE_TF32 (S = Q K^T from f32 Q "
                               "and K as tf32 operands, P and V bf16)"}

    # ---- end to end through the public API with host buffers ----------------
    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        h_q = q.cpu().pin_memory()
        h_sel, h_bt, h_cu = pin(w.selected), pin(w.block_tables), pin(w.cu_seqlens_q)
        h_used = pin(w.used_kv_lens) if w.pass_used else None
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_sel, h_bt, h_cu, h_used)
                  if t is not None)
        d2h = h_out.numel() * 4 + h_lse.numel() * 4
        d_q, d_sel, d_bt, d_cu = (torch.empty_like(x, device=dev) for x in (h_q, h_sel, h_bt, h_cu))
        d_used = torch.empty_like(h_used, device=dev) if h_used is not None else None
        n_e2e = min(args.steps, 300)
        s0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        s1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        for it in range(n_e2e + 3):
            timed = it >= 3
            flush.fill_(float(it))
            if timed:
                s0[it - 3].record(stream)
            d_q.copy_(h_q, non_blocking=True)
            d_sel.copy_(h_sel, non_blocking=True)
            d_bt.copy_(h_bt, non_blocking=True)
            d_cu.copy_(h_cu, non_blocking=True)
            if d_used is not None:
                d_used.copy_(h_used, non_blocking=True)
            sa.sa_attention(d_q, k, v, d_sel, w.cu_seqlens_q, d_cu, d_used, d_bt, w.hq, w.hkv,
                            w.head_dim, w.block_size, w.page_size, w.softmax_scale, w.causal,
                            split_edges=split, index=index, partials=partials, out=out,
                            lse=lse)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)
            if timed:
                s1[it - 3].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = sum(a.elapsed_time(b) for a, b in zip(s0, s1))
        e2e = {"value": w.tq * n_e2e / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": n_e2e}
        del h_q, h_out, h_lse, d_q, d_sel, d_bt, d_cu, d_used

    # ---- aggregate over ranks -----------------------------------------------
    elapsed_s, e2e_total = aggregate_ranks(total_ms / 1e3, e2e["value"] if e2e else None, world,
                                           dev)
    if e2e is not None:
        e2e["value"] = e2e_total
    del q, k, v, sel, cu, used, bt, flush, out, lse, index, partials, o_p, m_p, l_p
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    if rank != 0:
        return None, w

    peak, peak_kind = measured_peak()
    ms_per_step = elapsed_s * 1e3 / args.steps
    fwd_gbs = acct["forward"] / (fwd_ms / 1e3) / 1e9
    step_gbs = acct["step"] / (ms_per_step / 1e3) / 1e9
    kv_gbs = acct["kv"] / (ms_per_step / 1e3) / 1e9
    fwd_file = fwd_kernel.replace("_kernel", ".cu")
    traffic = ncu_traffic(fwd_file, name.replace("_ncu", "") +
                          ("_bf16p" if args.partials == "bf16" and not fused else ""))
    value = job_throughput(w.tq, args.steps, world, elapsed_s)
    dtype = "f32" if w.kv_dtype == "f32" else "bf16-kv/f32"
    rec = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {
            "workload": name, "batch": w.batch, "tq": w.tq, "hq": w.hq, "hkv": w.hkv,
            "head_dim": w.head_dim, "page_size": w.page_size, "block_size": w.block_size,
            "topk": w.topk, "max_pages": w.max_pages, "num_pages": w.num_pages,
            "kv_dtype": w.kv_dtype, "causal": w.causal, "split_edges": split,
            "o_partials": args.partials,
            "l2": "flushed before every timed step (512 MiB write, outside the step events)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "selected_kv_gbs": kv_gbs,
        "step_algorithmic_gbs": step_gbs,
        "step_frac_of_hbm": step_gbs / peak,
        "tflops": acct["flops"] / (ms_per_step / 1e3) / 1e12,
        "stages_ms": ({"index": index_ms, "forward_combine": fwd_ms} if fused else
                      {"index": index_ms, "forward": fwd_ms, "combine": comb_ms}),
        "roofline": {"kernel": f"{fwd_kernel} ({'sa_forward_combine' if fused else 'sa_forward'}"
                               + (", timed with its Q rounding pass)"
                                  if fwd_kernel == "forward_tc_kernel" else ")"),
                     "bound": "hbm",
                     "achieved": fwd_gbs, "peak": peak, "unit": "GB/s",
                     "frac": fwd_gbs / peak, "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": acct["forward"],
                     "traffic": traffic},
        "tensor_core_operands": "bf16" if fwd_kernel == "forward_tc_kernel" else None,
        "tf32_scores": tf32_scores,
        "algorithmic_bytes": {k_: acct[k_] for k_ in ("kv", "q", "partials_write", "out",
                                                       "step", "forward", "combine")},
        "edges": acct["edges"],
        "e2e": e2e,
        # library kernels per step: on the fused decode path the clear of the
        # build's counters, then the index kernel beside the fused decode
        # kernel; otherwise the index kernel, forward and combine (the
        # tensor-core forward preceded by the pass that rounds Q to bf16 into
        # its scratch and the two that build its longest-first work list)
        "gpu_launches": (3 if fused else (6 if fwd_kernel == "forward_tc_kernel" else 3))
                        * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    return rec, w


def run_ours(args, rank, world, local_rank):
    names = ([HEADLINE, *SUB_WORKLOADS] if args.workload == "all" else [args.workload])
    records, workloads = [], []
    for name in names:
        rec, w = measure_workload(name, args, rank, world, local_rank)
        records.append(rec)
        workloads.append(w)
    if rank != 0:
        return None
    # the oracle on the host cores, after every GPU timing (rank 0, N = 1 only)
    for rec, w in zip(records, workloads):
        rec["cpu_baseline"] = (cpu_baseline(w, args)
                               if world == 1 and not args.no_cpu_baseline else None)
    head = records[0]
    if len(records) > 1:
        head["sub_records"] = records[1:]
    return head


# --------------------------------------------------------------------------- oracle timing


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def oracle_threads() -> int:
    return max(1, min(os.cpu_count() or 1, 64))


def shard_costs(w, row_block):
    """The workload cut into independent shards (sequence b, kv head h, query
    rows [a, a + n) of b), each with an estimate of its oracle work: the
    multiply-adds of its kept entries' blocks (two per key and dimension, per
    GPU lane)."""
    cu = w.cu_seqlens_q
    shards = []
    for b in range(w.batch):
        qo = int(cu[b + 1] - cu[b])
        if qo == 0:
            continue
        lk = max(int(w.used_kv_lens[b]), 0) if w.pass_used else w.msb * w.block_size
        step = qo if qo <= row_block else row_block
        for h in range(w.hkv):
            for a in range(0, qo, step):
                n = min(step, qo - a)
                sel = w.selected[int(cu[b]) + a:int(cu[b]) + a + n, h]
                kept = int(np.sum((sel >= 0) & (sel.astype(np.int64) * w.block_size < lk)))
                cost = kept * w.qhead * w.block_size * w.head_dim * 2
                shards.append((b, h, a, n, cost))
    return shards


def make_shard(w, b, h, a, n):
    """Oracle inputs of one shard: queries [a, a + n) of sequence b against kv
    head h alone (q-heads h * qhead .. h * qhead + qhead - 1), with only the
    pages its kept blocks touch.  Under the right-aligned causal rule a
    sub-range of a sequence's queries is posed as a sequence of n queries whose
    KV length is lk - qo + a + n: each query's limit lk - qo + t is unchanged,
    so its output is too (blocks past the limit would be fully masked)."""
    import inputs

    cu = w.cu_seqlens_q
    qo = int(cu[b + 1] - cu[b])
    lk = max(int(w.used_kv_lens[b]), 0) if w.pass_used else w.msb * w.block_size
    if n < qo and w.causal:
        assert lk >= qo, "sub-ranges need lk >= qo under the causal rule"
        lk_sub = lk - qo + a + n
    else:
        lk_sub = lk
    rows = np.arange(int(cu[b]) + a, int(cu[b]) + a + n)
    sel = np.ascontiguousarray(w.selected[rows][:, h:h + 1, :])
    d, qh = w.head_dim, w.qhead
    qidx = ((rows[:, None] * w.hq + h * qh) * d + np.arange(qh * d)[None, :]).astype(np.uint64)
    q = inputs.counter_normal_at(w.seed, inputs.STREAM_Q, qidx).reshape(n, qh, d)
    blocks = np.unique(sel[(sel >= 0) & (sel.astype(np.int64) * w.block_size < lk_sub)])
    bt_row = w.block_tables[b].astype(np.int64)
    cols = (blocks[:, None].astype(np.int64) * w.ppb + np.arange(w.ppb)[None, :]).ravel()
    pages = np.unique(bt_row[cols][bt_row[cols] >= 0])
    pos = np.searchsorted(pages, bt_row)
    hit = (bt_row >= 0) & (pos < pages.size)
    hit[hit] = pages[pos[hit]] == bt_row[hit]
    bt = np.where(hit, pos, -1).astype(np.int32)[None, :]
    pe, hs = w.page_elems, w.page_size * d

    def pool(stream):
        if pages.size == 0:
            vals = np.zeros((1, 1, w.page_size, d), np.float32)
        else:
            idx = (pages[:, None] * pe + h * hs + np.arange(hs)[None, :]).astype(np.uint64)
            vals = inputs.counter_normal_at(w.seed, stream, idx).reshape(pages.size, 1,
                                                                         w.page_size, d)
        return inputs.bf16_bits(vals) if w.kv_dtype == "bf16" else vals

    return {"q": q, "k": pool(inputs.STREAM_K), "v": pool(inputs.STREAM_V), "sel": sel, "bt": bt,
            "cu": np.array([0, n], np.int64),
            "used": np.array([lk_sub], np.int32) if (w.pass_used or lk_sub != lk) else None,
            "hq": qh, "queries": n / w.hkv}


def pick_shards(w, budget_macs, row_block, rng_seed=0):
    """Shards in a seeded random order until their estimated work reaches
    budget_macs (at least one)."""
    shards = shard_costs(w, row_block)
    order = np.random.default_rng(rng_seed).permutation(len(shards))
    picked, acc = [], 0
    for j in order:
        picked.append(shards[j])
        acc += shards[j][4]
        if acc >= budget_macs:
            break
    return picked


def assign_lpt(shards, threads):
    """Longest-first assignment of shards to threads (by estimated cost)."""
    bins = [[] for _ in range(threads)]
    load = [0] * threads
    for s in sorted(shards, key=lambda s: -s[4]):
        t = int(np.argmin(load))
        bins[t].append(s)
        load[t] += s[4]
    return [b for b in bins if b]


def run_oracle_phases(w, groups, pool, phases=("index", "partials_combine", "direct")):
    """Run the oracle over prepared shard groups (one group per thread), one
    phase at a time; returns wall seconds per phase."""
    import oracle

    state = [[None] * len(g) for g in groups]

    def index_part(t):
        for j, s in enumerate(groups[t]):
            state[t][j] = oracle.build_index(s["sel"], s["cu"], s["used"], w.max_pages,
                                             w.block_size, w.page_size, 0)

    def fwd_part(t):
        for j, s in enumerate(groups[t]):
            idx = state[t][j]
            o, m, l = oracle.forward(s["q"], s["k"], s["v"], idx, s["bt"], s["cu"], s["used"],
                                     s["hq"], w.head_dim, w.softmax_scale, w.causal)
            oracle.combine(idx, s["hq"], w.head_dim, o, m, l)

    def direct_part(t):
        for s in groups[t]:
            oracle.direct(s["q"], s["k"], s["v"], s["sel"], s["bt"], s["cu"], s["used"],
                          s["hq"], w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                          w.causal)

    fns = {"index": index_part, "partials_combine": fwd_part, "direct": direct_part}
    walls = {}
    for ph in phases:
        t0 = time.perf_counter()
        list(pool.map(fns[ph], range(len(groups))))
        walls[ph] = time.perf_counter() - t0
    return walls


CALIB_NS_PER_MAC = 2.5       # single-thread oracle speed, for sizing the samples only


def oracle_sample(w, wall_s, threads, seed=0):
    """Prepared shard groups whose partials phase should take about wall_s
    seconds on `threads` host threads."""
    import oracle

    oracle.build()
    row_block = 32 if w.tq > 2 * w.batch else 1
    budget = wall_s * threads / (CALIB_NS_PER_MAC * 1e-9)
    shards = pick_shards(w, budget, row_block, seed)
    groups_meta = assign_lpt(shards, threads)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        groups = list(ex.map(lambda g: [make_shard(w, b, h, a, n) for (b, h, a, n, _) in g],
                             groups_meta))
    queries = sum(s["queries"] for g in groups for s in g)
    desc = (f"{len(shards)} shard(s) (sequence, kv head, query rows) in a seeded random order, "
            f"{queries:g} query-equivalents (query x kv head / hkv)")
    return groups, queries, desc


def cpu_baseline(w, args):
    """The oracle timed on the host cores: index, partials + combine, and the
    query-outer direct attention, each as queries/s over the same sample;
    `value` is the path (index + partials + combine)."""
    threads = oracle_threads()
    groups, queries, desc = oracle_sample(w, args.cpu_seconds, threads)
    with cf.ThreadPoolExecutor(max_workers=len(groups)) as ex:
        walls = run_oracle_phases(w, groups, ex)
    path_s = walls["index"] + walls["partials_combine"]
    return {"value": queries / path_s, "unit": UNIT, "cores": len(groups), "kind": "oracle",
            "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
            "rates": {ph: queries / s for ph, s in walls.items()},
            "sample": f"{desc}; one host thread per core, f64"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step runs the index and the
    partials + combine over one bounded sample of the workload on the host
    cores (rank 0 only)."""
    if rank != 0:
        return None
    workload = HEADLINE if args.workload == "all" else args.workload
    w = make_workload(workload, args.seed)
    threads = oracle_threads()
    per_step = getattr(args, "ref_step_seconds", 1.0)
    groups, queries, desc = oracle_sample(w, per_step, threads)
    phases = ("index", "partials_combine")
    with cf.ThreadPoolExecutor(max_workers=len(groups)) as ex:
        for _ in range(args.warmup):
            run_oracle_phases(w, groups, ex, phases)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run_oracle_phases(w, groups, ex, phases)
        el = time.perf_counter() - t0
    value = queries * args.steps / el
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "sample_queries_per_step": queries},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(groups), "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"{desc} per step; one host thread per core, f64"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if res is not None and rank == 0:
        print(json.dumps(res))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
