"""Benchmark: FlashMask-style masked attention, forward + backward, on the
128K long-context document-packing workload (B=1, H=8, N=131072, d=128,
log-normal documents, causal within each document).

One step = one pass of the hot path over the workload: tile classification,
forward, backward (preprocess, main, dQ postprocess).  The metric is TFLOP/s
on unmasked FLOPs (4d per attended (i, j) pair per head forward, 10d
backward, 14d together); `value` is the fwd+bwd figure with inputs resident
in HBM.  `e2e` repeats the step through the C ABI from pinned host buffers:
row-form mask conversion on the host, host-to-device copies of Q, K, V, dO
and the bounds, the device work, and device-to-host copies of O, lse, dQ,
dK, dV, all inside the timed region; the copies run on their own streams
with two buffer sets, so one step's copies overlap its neighbours' compute;
the figure is the median of three runs (the host links are shared with the
machine's other GPUs).  `e2e_bf16_outputs` repeats it with bf16 O, dQ, dK,
dV (half the bytes read back).  `graph` times the same step captured
once into a CUDA graph (fm_step_graph_create) and replayed, one launch per
step.  `fp8_fwd` times the forward on e4m3 inputs (fm_attn_fwd_fp8) and the
quantization of Q, K, V beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fm|reference]
Under torchrun every rank runs the whole workload on its own GPU (independent
replicas, weak scaling); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from long_context_fm_gb300 import workloads as W  # noqa: E402

METRIC = "fwd and fwd+bwd TFLOP/s on unmasked FLOPs (% of GB300 BF16 peak) at N=128K"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + written) per launch of the dominant kernel from a 1-pass
# ncu capture of dram__bytes_read.sum and dram__bytes_write.sum, keyed by the
# kernel, the hash of the source it was taken on (stale entries are ignored)
# and the workload.
NCU_TRAFFIC = {
    ("bwd", "63f8834e03518abe", "long_packing_128k"): 1649.403e6 + 1566.780e6,
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def src_hash(name):
    """Hash of a kernel's source, its PTX helpers and the classifier (whose
    work order decides which tiles run together, hence the DRAM traffic)."""
    csrc = os.path.join(ROOT, "long_context_fm_gb300", "csrc")
    h = hashlib.sha256()
    for f in (name, "fm_ptx.cuh", "fm_classify.cu"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
def attended_pairs_per_head(m, b, hm, N):
    """Attended pairs of one mask head, from interval arithmetic on the bounds."""
    l0, l1 = m["lts"][b, hm].astype(np.int64), m["lte"][b, hm].astype(np.int64)
    u0, u1 = m["uts"][b, hm].astype(np.int64), m["ute"][b, hm].astype(np.int64)
    ln, un = np.maximum(l1 - l0, 0), np.maximum(u1 - u0, 0)
    inter = np.where((ln > 0) & (un > 0), np.maximum(np.minimum(l1, u1) - np.maximum(l0, u0), 0), 0)
    return int((N - (ln + un - inter)).sum())


def total_pairs(wl, m):
    tot = 0
    for b in range(wl.B):
        for h in range(wl.H):
            tot += attended_pairs_per_head(m, b, h if wl.Hm == wl.H else 0, wl.N)
    return tot


def workload_of(args):
    """The named workload, with H overridden by --heads (a smaller case of the
    same mask for profiler captures; the default run never sets it)."""
    wl = W.FULL[args.config]
    return wl.with_(H=args.heads) if args.heads else wl


def precision_flags(args, wl):
    """FM_FLAG_PRECISE (1) or 0.  auto: precise for the x2-scaled prefix
    workloads, whose gradients of tens exceed the max-abs bound with one bf16
    rounding of P and dS (the mode their parity tests run in), standard for
    every other workload."""
    if args.precision == "auto":
        return 1 if wl.input_scale != 1.0 else 0
    return 1 if args.precision == "precise" else 0


def hbm_bytes(wl, nnz_tiles, o_bytes=4, g_bytes=4):
    """Algorithmic HBM bytes per launch of the memory-bound kernels: what each
    must read and write at least once.
      classify_minmax: 16 B of bounds per column read, 32 B of min/max per KV tile written
      classify_lists:  the min/max read once; labels (1 B per tile pair), 4 B per
                       non-skip pair in each of the two lists and 4 B per list count written
      classify_order:  the list counts read, the two orders written
      bwd_pre:         O and dO read, D (4 B per row) and the zeroed dQ accumulator written
      bwd_post:        the dQ accumulator read, dQ written"""
    S = wl.B * wl.Hm
    n_t = -(-wl.N // 128)
    rows = wl.B * wl.H * wl.N
    d = wl.d
    return {
        "classify_minmax": S * (16 * wl.N + 32 * n_t),
        "classify_lists": S * (32 * n_t + n_t * n_t + 8 * n_t) + 8 * nnz_tiles,
        "classify_order": S * 16 * n_t,
        "bwd_pre": rows * (o_bytes * d + 2 * d + 4 + 4 * d),
        "bwd_post": rows * (4 * d + g_bytes * d),
    }


def max_over_ranks(vals, world, device):
    """Element-wise max of per-rank timings (the only collective of the run)."""
    t = torch.tensor(vals, dtype=torch.float64)
    if world > 1:
        t = t.to(device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        t = t.cpu()
    return [float(x) for x in t]


def run_fm(args, rank, world, local_rank):
    from long_context_fm_gb300 import fm

    wl = workload_of(args)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    m = W.make_mask(wl)
    pairs = total_pairs(wl, m)
    d = wl.d
    fwd_flops = 4.0 * d * pairs
    bwd_flops = 10.0 * d * pairs
    # inputs on the device (values drawn on the device, seeded per rank)
    q, k, v, dO = W.make_inputs(wl, seed=1000 + rank, device=dev)
    B, H, N = wl.B, wl.H, wl.N
    stream = torch.cuda.current_stream(dev)
    bnd = [torch.from_numpy(np.ascontiguousarray(m[x])).to(dev) for x in ("lts", "lte", "uts", "ute")]
    bounds = fm.make_bounds(*bnd)
    plan = torch.empty(fm.fm_plan_bytes(B, wl.Hm, N), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3))
    ws = torch.empty(fm.fm_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    scale = wl.scale
    flags = precision_flags(args, wl)
    # non-skip (Q tile, KV tile) pairs: the classifier's list bytes
    labels = torch.empty((B, wl.Hm, -(-N // 128), -(-N // 128)), dtype=torch.uint8, device=dev)
    fm.fm_tile_classify(bounds, plan, status, labels=labels, stream=stream)
    nnz_tiles = int(torch.count_nonzero(labels).item())
    del labels

    def step():
        fm.fm_tile_classify(bounds, plan, status, stream=stream)
        fm.fm_attn_fwd(q, k, v, bounds, plan, scale, o, lse, status, stream=stream, flags=flags)
        fm.fm_attn_bwd(q, k, v, o, lse, dO, bounds, plan, scale, dq, dk, dv, ws, status, stream=stream,
                       flags=flags)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}: {fm.fm_status_string(int(status.item()))}")

    # ---- device-resident timed region
    barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fm.fm_profile_begin()
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    smi_id = (uuid if uuid.startswith("GPU-") else f"GPU-{uuid}") if uuid else str(local_rank)
    with ClockSampler(smi_id) as clocks:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    recs = fm.fm_profile_end()
    barrier()
    ms_total = ev0.elapsed_time(ev1)
    ms_step = ms_total / args.steps
    per_kernel = {}
    for name, ms in recs:
        per_kernel.setdefault(name, []).append(ms)
    avg = {kname: sum(v_) / len(v_) for kname, v_ in per_kernel.items()}
    launches = len(recs)

    # ---- the same step replayed from a captured graph (one launch per step)
    gh = fm.fm_step_graph_create(q, k, v, dO, bounds, plan, scale, o, lse, status, dq, dk, dv, ws, flags)
    for _ in range(2):
        fm.fm_step_graph_launch(gh, stream)
    torch.cuda.synchronize(dev)
    barrier()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        fm.fm_step_graph_launch(gh, stream)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = g0.elapsed_time(g1) / args.steps
    fm.fm_step_graph_destroy(gh)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in graph replay")

    # ---- FP8 forward: e4m3 Q, K, V^T (per-tensor scales); the forward timed
    # alone, and one quantization of Q, K, V timed beside it
    fp8 = None
    if d == 128 and N % 16 == 0:
        q8, dq8 = fm.fm_quantize_fp8(q, stream=stream)
        k8, dk8 = fm.fm_quantize_fp8(k, stream=stream)
        vt8, dv8 = fm.fm_quantize_fp8(v, transpose=True, stream=stream)
        descale = torch.cat([dq8, dk8, dv8])
        o8 = torch.empty_like(o)

        def fwd8():
            fm.fm_attn_fwd_fp8(q8, k8, vt8, descale, bounds, plan, scale, o8, lse, status, stream=stream)

        for _ in range(max(args.warmup, 2)):
            fwd8()
        torch.cuda.synchronize(dev)
        f0, f1, f2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        f0.record(stream)
        for _ in range(args.steps):
            fwd8()
        f1.record(stream)
        for _ in range(args.steps):
            fm.fm_quantize_fp8(q, out=q8, descale=dq8, stream=stream)
            fm.fm_quantize_fp8(k, out=k8, descale=dk8, stream=stream)
            fm.fm_quantize_fp8(v, transpose=True, out=vt8, descale=dv8, stream=stream)
        f2.record(stream)
        torch.cuda.synchronize(dev)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the FP8 forward")
        fp8 = (f0.elapsed_time(f1) / args.steps, f1.elapsed_time(f2) / args.steps)

    # ---- end to end through the C ABI from pinned host buffers, pipelined:
    # host-to-device copies, the step and device-to-host copies run on three
    # streams with two buffer sets, so the copies of one step overlap the
    # compute of its neighbours; every step still copies its own inputs in and
    # its own outputs out inside the timed region.
    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, dO))
    rows = m["rows"]
    multi = m["row_intervals"]

    def run_e2e(out_dtype):
        """Pipelined end-to-end steps with O, dQ, dK, dV of out_dtype (lse fp32);
        returns seconds per step and the bytes copied in and out per step."""
        def device_set():
            st = dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v), dO=torch.empty_like(dO),
                      lse=torch.empty_like(lse), bnd=[torch.empty_like(b_) for b_ in bnd])
            for key in ("o", "dq", "dk", "dv"):
                st[key] = torch.empty(q.shape, dtype=out_dtype, device=dev)
            st["bounds"] = fm.make_bounds(*st["bnd"])
            return st

        sets = [device_set(), device_set()]
        host_out = [dict((key, torch.empty_like(sets[0][key], device="cpu").pin_memory())
                         for key in ("o", "lse", "dq", "dk", "dv")) for _ in range(2)]
        host_bnd = [[torch.empty(bnd[0].shape, dtype=torch.int32).pin_memory() for _ in range(4)] for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo)) + 4 * bnd[0].numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
        s_h2d, s_cmp, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_h2d = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_d2h = [torch.cuda.Event() for _ in range(2)]

        def e2e_issue(i):
            sidx = i % 2
            bs, hb = sets[sidx], host_bnd[sidx]
            if rows is not None:                                     # host conversion of the row form
                cols = fm.fm_mask_from_rows(*rows)
            elif multi is not None:                                  # several intervals per row
                cols = fm.fm_mask_from_row_intervals(*multi)
            else:
                cols = [m[x] for x in ("lts", "lte", "uts", "ute")]
            if i >= 2:
                ev_h2d[sidx].synchronize()                           # hb is still being copied from
            for dst, src in zip(hb, cols):
                dst.numpy()[...] = src
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(ev_cmp[sidx])                   # the set's inputs are free again
                for dst, src in zip(bs["bnd"], hb):
                    dst.copy_(src, non_blocking=True)
                for key, src in zip(("q", "k", "v", "dO"), (hq, hk, hv, hdo)):
                    bs[key].copy_(src, non_blocking=True)
                ev_h2d[sidx].record(s_h2d)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_h2d[sidx])
                if i >= 2:
                    s_cmp.wait_event(ev_d2h[sidx])                   # the set's outputs have been read out
                fm.fm_tile_classify(bs["bounds"], plan, status, stream=s_cmp)
                fm.fm_attn_fwd(bs["q"], bs["k"], bs["v"], bs["bounds"], plan, scale, bs["o"], bs["lse"], status,
                               stream=s_cmp, flags=flags)
                fm.fm_attn_bwd(bs["q"], bs["k"], bs["v"], bs["o"], bs["lse"], bs["dO"], bs["bounds"], plan, scale,
                               bs["dq"], bs["dk"], bs["dv"], ws, status, stream=s_cmp, flags=flags)
                ev_cmp[sidx].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_cmp[sidx])
                for key, dst in host_out[sidx].items():
                    dst.copy_(bs[key], non_blocking=True)
                ev_d2h[sidx].record(s_d2h)

        torch.cuda.synchronize(dev)
        for i in range(2):
            e2e_issue(i)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_steps = max(2, min(args.steps, 8))
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_issue(i + 2)
        torch.cuda.synchronize(dev)
        barrier()
        sec = (time.perf_counter() - t0) / e2e_steps
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the end-to-end steps")
        del sets
        return sec, h2d, d2h

    # The host links are shared with the machine's other GPUs, so one short run
    # varies by tens of percent: three runs of each output type, alternating,
    # and the median of each.
    runs32, runs16 = [], []
    for _ in range(3):
        runs32.append(run_e2e(torch.float32))
        runs16.append(run_e2e(torch.bfloat16))
    e2e_s, h2d, d2h = sorted(runs32)[1]
    e2e16_s, _, d2h16 = sorted(runs16)[1]

    ms_step, e2e_s, e2e16_s, graph_ms = max_over_ranks([ms_step, e2e_s, e2e16_s, graph_ms], world, dev)
    return dict(wl=wl, pairs=pairs, fwd_flops=fwd_flops, bwd_flops=bwd_flops, ms_step=ms_step,
                avg=avg, launches=launches, clocks=clocks.summary(), e2e_s=e2e_s, h2d=h2d, d2h=d2h,
                e2e16_s=e2e16_s, d2h16=d2h16, graph_ms=graph_ms, fp8=fp8, flags=flags, nnz_tiles=nnz_tiles)


def mask_description(wl):
    p = wl.params
    return {
        "causal": "causal",
        "docs_uniform": f"documents of uniform length in [{p.get('lo')}, {p.get('hi')}], causal within document",
        "docs_lognormal": (f"log-normal documents (median {p.get('median')}, sigma {p.get('sigma')}, "
                           f"clip [{p.get('lo')}, {p.get('hi')}]), causal within document"),
        "window": f"causal sliding window of {p.get('window')} keys",
        "window_sink": f"causal sliding window of {p.get('window')} keys plus {p.get('sink')} sink keys",
        "prefix": f"prefix LM: bidirectional prefix of {p.get('prefix')}, causal after it",
        "prefix_random": (f"prefix of {p.get('prefix')} plus a random lower masked range per column "
                          "(lts uniform in [j, N])"),
    }.get(wl.mask, wl.mask)


def l2_note(wl):
    gib = 4 * wl.B * wl.H * wl.N * wl.d * 2 / 2 ** 30
    if gib * 2 ** 30 > 129e6:
        return f"inputs larger than L2 (Q, K, V, dO {gib:.2f} GiB), no flush"
    return f"inputs of {gib * 1024:.0f} MiB (Q, K, V, dO) may stay in the 129 MB L2: no flush"


def cpu_baseline_sample(wl, m, max_docs=3, rows=4096):
    """The oracle, as it stands, on an independent sub-problem of head 0 of
    the same workload: the first documents when the mask is document packing
    (causal within each document, nothing across documents), else the mask
    restricted to the leading `rows` x `rows` block."""
    import oracle

    if m["docs"] is not None:
        docs = m["docs"][0]
        S = int(sum(docs[:max_docs]))
        what = "the first document of head 0" if max_docs == 1 else f"the first {max_docs} documents of head 0"
    else:
        S = min(wl.N, rows)
        what = f"the leading {S} x {S} block of head 0's mask"
    sub = {x: np.minimum(m[x][:1, :1, :S], S).astype(np.int32) for x in ("lts", "lte", "uts", "ute")}
    # attended (i, j) pairs of the sub-problem: per column, S minus the rows of
    # the union of its two masked ranges
    l0, l1, u0, u1 = (sub[x][0, 0].astype(np.int64) for x in ("lts", "lte", "uts", "ute"))
    ln, un = np.maximum(l1 - l0, 0), np.maximum(u1 - u0, 0)
    inter = np.where((ln > 0) & (un > 0), np.maximum(np.minimum(l1, u1) - np.maximum(l0, u0), 0), 0)
    pairs = int((S - (ln + un - inter)).sum())
    g = torch.Generator().manual_seed(0)
    q, k, v, dO = (torch.randn(1, 1, S, wl.d, generator=g).to(torch.bfloat16) for _ in range(4))
    t0 = time.perf_counter()
    oracle.forward(q, k, v, sub, wl.scale)
    oracle.backward(q, k, v, dO, sub, wl.scale)
    dt = time.perf_counter() - t0
    tflops = 14.0 * wl.d * pairs / dt / 1e12
    return dict(value=tflops, unit="TFLOP/s", cores=oracle.num_threads(), kind="oracle", what=what,
                sample=f"fp64 oracle fwd+bwd on {what} ({S} rows, {pairs} attended pairs), {dt:.1f} s")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fm", choices=["fm", "reference"])
    ap.add_argument("--config", default="long_packing_128k", choices=list(W.FULL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the workload's head count (a smaller case of the same mask, for ncu captures)")
    ap.add_argument("--precision", default="auto", choices=["auto", "standard", "precise"],
                    help="standard: bf16 P and dS operands; precise: split-bf16 P and dS (FM_FLAG_PRECISE); "
                         "auto: precise for the x2-scaled prefix workloads, standard otherwise")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workload_of(args)

    if args.impl == "reference":
        if rank != 0:
            return
        m = W.make_mask(wl)
        for _ in range(args.warmup):
            cpu_baseline_sample(wl, m, max_docs=1)
        vals = [cpu_baseline_sample(wl, m, max_docs=1) for _ in range(args.steps)]
        cb = vals[-1]
        val = statistics.median(v_["value"] for v_ in vals)
        line = {"metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d,
                           "sample": f"{cb['what']} per step"},
                "cpu_baseline": {k_: cb[k_] for k_ in ("kind", "cores", "sample")} | {"value": val, "unit": "TFLOP/s"},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    r = run_fm(args, rank, world, local_rank)
    if rank == 0:
        peaks, src = load_peaks()
        fwd_ms = r["avg"].get("fwd", float("nan"))
        bwd_ms = r["avg"].get("bwd", float("nan"))
        step_flops = r["fwd_flops"] + r["bwd_flops"]
        value = world * step_flops / (r["ms_step"] * 1e-3) / 1e12
        fwd_tflops = r["fwd_flops"] / (fwd_ms * 1e-3) / 1e12
        bwd_tflops = r["bwd_flops"] / (bwd_ms * 1e-3) / 1e12
        peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        peak_hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        key = src_hash("fm_bwd.cu")
        traffic = NCU_TRAFFIC.get(("bwd", key, wl.name))
        fwd_bwd_tflops = value / world

        def fracs(x):
            return {"burst": x / peak_burst, "sustained": x / peak_sus}

        # The kernels are timed inside a step of a few milliseconds (a timed
        # region well under a second): the burst peak is the one that applies;
        # the sustained figure is given beside it.
        hbm = {}
        for kname, nbytes in hbm_bytes(wl, r["nnz_tiles"]).items():
            ms = r["avg"].get(kname)
            if ms:
                gbs = nbytes / (ms * 1e-3) / 1e9
                hbm[kname] = {"bytes": nbytes, "ms": ms, "GB/s": gbs, "frac": gbs / peak_hbm}
        precise = r["flags"] == 1
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": r["wl"].name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d,
                       "mask": mask_description(wl),
                       "attended_pairs": r["pairs"], "outputs": "fp32 O, dQ, dK, dV",
                       "precision": ("precise (split-bf16 P and dS tensor-core operands, fp32 accumulation)"
                                     if precise else
                                     "standard (bf16 P and dS tensor-core operands, fp32 accumulation)"),
                       "l2": l2_note(wl)},
            "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
            "frac_of_peak": {"fwd": fracs(fwd_tflops), "bwd": fracs(bwd_tflops), "fwd_bwd": fracs(fwd_bwd_tflops),
                             "peaks": f"{src}: bf16 burst {peak_burst}, sustained {peak_sus} TFLOP/s"},
            "kernel_ms": r["avg"],
            "hbm": {"peak_GB/s": peak_hbm, "peak_source": f"{src} copy bandwidth", "kernels": hbm},
            "roofline": {"kernel": "fm_bwd_kernel", "bound": "tensor", "achieved": bwd_tflops,
                         "peak": peak_burst, "unit": "TFLOP/s", "frac": bwd_tflops / peak_burst,
                         "traffic": traffic, "peak_source": f"{src} bf16 burst",
                         "frac_of_sustained": bwd_tflops / peak_sus},
            "gpu_launches": r["launches"],
            "fp8_fwd": None if r["fp8"] is None else {
                "ms": r["fp8"][0], "value": world * r["fwd_flops"] / (r["fp8"][0] * 1e-3) / 1e12, "unit": "TFLOP/s",
                "quantize_qkv_ms": r["fp8"][1],
                "note": "e4m3 Q, K, V^T with per-tensor scales, P rounded to e4m3; forward alone, same FLOPs"},
            "graph": {"ms_per_step": r["graph_ms"], "value": world * step_flops / (r["graph_ms"] * 1e-3) / 1e12,
                      "unit": "TFLOP/s", "launches_per_step": 1,
                      "note": "the same step captured once (fm_step_graph_create) and replayed"},
            "clocks": r["clocks"],
            "e2e": {"value": world * step_flops / r["e2e_s"] / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "e2e_bf16_outputs": {"value": world * step_flops / r["e2e16_s"] / 1e12, "unit": "TFLOP/s",
                                 "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h16"],
                                 "note": "the same end-to-end step with bf16 O, dQ, dK, dV (lse fp32)"},
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = {k_: v_ for k_, v_ in cpu_baseline_sample(wl, W.make_mask(wl), max_docs=7).items()
                                    if k_ != "what"}
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
