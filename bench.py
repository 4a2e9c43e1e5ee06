"""Benchmark of paged-attention decode on GB300 -- one JSON line on rank 0.

A step is one pass of the whole decode path (plan -> tile kernel -> partition
reduce) over the long-context decode workload, both KV variants of it:
MXFP4 (e2m1 + e8m0 per 32) and fp8 e4m3 with per-token scales; batch 16, 1 KV
head, GQA 16, head_dim 128, page 128, qlen 1, context lengths uniform in
[120000, 131072], bf16 query and output.  Inputs are synthetic and seeded, resident
in HBM before the timed region; each call streams 273 MB / 530 MB of KV, more
than the 129 MB L2, so no flush is needed between steps.

value  = algorithmic bytes of the step (owned-token KV + scales + Q + O + table)
         / device time of the step, in GB/s, summed over ranks (replicas).
e2e    = the same metric through the C ABI with host buffers: per step the query,
         block tables and context lengths are copied from pinned host memory and
         the output is copied back, inside the timed region (the KV cache is the
         engine's resident state and stays in HBM); the copies run on a second stream,
         double-buffered, overlapping the neighbouring steps' compute.
per_config = every workload of the method, timed one call at a time through the C ABI
         (plan + tile + reduce, device buffers) with the 129 MB L2 flushed before each
         call: µs/call, GB/s of algorithmic bytes and the fraction of the HBM peak; also
         the same call replayed from a CUDA graph, tile + reduce on a plan built
         beforehand (us_planned), and the whole call with one partition per
         unit, rows written directly and no reduce (us_one_partition).
roofline = the tile kernel with the largest share of the step, against the measured HBM
         peak; roofline.variants gives, per long-context variant, its tile kernel and its
         whole call (pa_decode_run: plan + tile + reduce) in µs and as a fraction of the
         peak -- one call at a time (call_us) and calls back to back.  The roofline
         object closes the line.
--impl reference times the fp64 CPU oracle on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_attention_decode_02_gb300 import ops, replicas, synth  # noqa: E402

METRIC = "pa_decode µs/call and achieved KV GB/s (fraction of GB300 HBM peak)"
WORKLOAD = ("long-context decode, MXFP4 + fp8/token KV, B16 Hkv1 G16 D128 page128 qlen1 "
                  "L~U[120000,131072]")
FALLBACK_HBM_GBS = 6800.0
KERNEL = None  # decode kernel choice passed to every call (--kernel)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="pa_bench_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        except OSError:
            return None
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def tile_kernel_name(case) -> str:
    """The decode kernel a call of this workload launches (the library's own choice)."""
    if KERNEL == "tc":
        return "pa_tc_kernel"
    if case.kv == synth.KV_MXFP4 and KERNEL is None:
        return "pa_mx_kernel"
    return "pa_tile_kernel"


def traffic_from_profile(kernel: str):
    """dram bytes per launch of this kernel on the long-context workload, from the committed
    ncu summary profiles/ncu_traffic_<kernel>.txt, or None when there is none or the kernel
    sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"ncu_traffic_{kernel}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if "=" in line and not line.startswith("#"):
            k, v = line.strip().split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def _code_only(text: str) -> str:
    """C / CUDA source without comments, trailing blanks or empty lines: what the compiler
    sees, so that an edit of comments alone does not change the hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c in "\"'":  # string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(csrc=None):
    """sha256 (first 16 hex) over the kernel sources, comments removed."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "paged_attention_decode_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def per_config(device, peak, calls=10, warmup=3):
    """µs/call and GB/s of every workload of the method, one call at a time, L2 flushed:
    the whole call (plan, decode, reduce), the same call replayed from a CUDA graph, and
    decode + reduce on a plan built beforehand (a model plans once per step and reuses the
    plan in every layer; the pages' "planned" timings take the plan as an input too)."""
    cases = [synth.config1(), synth.config2("a"), synth.config2("b"), synth.config3(qlen=1),
             synth.config3(qlen=4)] + [synth.config4(batch=b) for b in (8, 32, 64, 128, 256, 512, 4096)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    res = {}
    for case in cases:
        p = synth.make(case, device=device)
        q = p["query"]
        if q.dtype == torch.uint8:
            q = q.view(torch.float8_e4m3fn)
        out = torch.empty(tuple(p["query"].shape), dtype=torch.bfloat16, device=device)
        args = ops.make_args(q, p["key_cache"], p["value_cache"], p["block_tables"], p["context_lens"],
                             out, key_scale=p["key_scale"], value_scale=p["value_scale"],
                             q_scale=p["q_scale"], softmax_scale=case.scale_qk(), kernel=KERNEL)
        ws = ops.alloc_workspace(args, device)
        # one partition per unit (the pages' plan-free mode): rows written directly, no reduce
        args1 = ops.make_args(q, p["key_cache"], p["value_cache"], p["block_tables"],
                              p["context_lens"], out, key_scale=p["key_scale"],
                              value_scale=p["value_scale"], q_scale=p["q_scale"],
                              softmax_scale=case.scale_qk(), max_partitions=1, kernel=KERNEL)
        ws1 = ops.alloc_workspace(args1, device)
        for _ in range(warmup):
            ops.pa_decode_run(args, ws, stream)
            ops.pa_decode_run(args1, ws1, stream)
        # the same call captured once in a CUDA graph (how a serving loop issues it)
        gs = torch.cuda.Stream(device)
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            ops.pa_decode_run(args, ws, gs)
            with torch.cuda.graph(graph, stream=gs):
                ops.pa_decode_run(args, ws, gs)
        stream.wait_stream(gs)
        torch.cuda.synchronize()
        def planned():
            ops.pa_decode(args, ws, stream)
            ops.pa_decode_reduce(args, ws, stream)

        ts, tg, tp, tf = [], [], [], []
        for _ in range(calls):
            for launch, acc in ((lambda: ops.pa_decode_run(args, ws, stream), ts),
                                (graph.replay, tg), (planned, tp),
                                (lambda: ops.pa_decode_run(args1, ws1, stream), tf)):
                if launch is planned:  # (small workloads run pa_decode_run as one launch
                    ops.pa_decode_plan(args, ws, stream)  # that leaves no plan behind)
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
                torch.cuda.synchronize()
                acc.append(e0.elapsed_time(e1))
        assert ops.pa_decode_read_status(ws) == 0 and ops.pa_decode_read_status(ws1) == 0, case.name
        nbytes = synth.algorithmic_bytes(case, p["context_lens"].cpu().tolist())
        med, medg, medp = statistics.median(ts), statistics.median(tg), statistics.median(tp)
        medf = statistics.median(tf)
        res[case.name] = {"us": round(med * 1e3, 2), "us_graph": round(medg * 1e3, 2),
                     "us_planned": round(medp * 1e3, 2), "us_one_partition": round(medf * 1e3, 2),
                     "bytes": nbytes, "GBps": round(nbytes / (med * 1e-3) / 1e9, 1),
                     "frac": round(nbytes / (med * 1e-3) / 1e9 / peak, 4)}
        del graph
        del p, out, ws, ws1
    res.update(kv_write_config(device, peak, calls))
    del flush
    torch.cuda.empty_cache()
    return res


def kv_write_config(device, peak, calls):
    """The MXFP4 KV-cache write (include/pa_kv_write.h): 65536 new tokens x 8 KV heads x
    head_dim 128, K and V, scattered over the slots of a paged cache; bytes = bf16 rows read
    + e2m1 data and e8m0 scales written + the slot map.  The 268 MB of rows read are twice
    the L2, so calls run back to back without a flush (a flush by writing would leave L2
    full of dirty lines, whose write-back this write-heavy kernel would pay for)."""
    T, Hkv, D, S = 65536, 8, 128, 128
    NB = T // S + 1
    g = torch.Generator().manual_seed(4242)
    key = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16).to(device)
    value = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16).to(device)
    slots = (torch.randperm(T, generator=g) + S).to(torch.int64).to(device)  # block 0 unused
    kc = torch.zeros((NB, Hkv, S, D // 2), dtype=torch.uint8, device=device)
    vc = torch.zeros_like(kc)
    ks = torch.zeros((NB, Hkv, S, D // 32), dtype=torch.uint8, device=device)
    vs = torch.zeros_like(ks)
    args = ops.mxfp4_write_args(key, value, slots, kc, vc, ks, vs)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        ops.mxfp4_kv_write(args, stream)
    ts = []
    for _ in range(calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ops.mxfp4_kv_write(args, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    med = statistics.median(ts)
    nbytes = 2 * T * Hkv * (2 * D + D // 2 + D // 32) + 8 * T
    return {"mxfp4_kv_write_t65536_h8_d128": {
        "us": round(med * 1e3, 2), "bytes": nbytes,
        "GBps": round(nbytes / (med * 1e-3) / 1e9, 1),
        "frac": round(nbytes / (med * 1e-3) / 1e9 / peak, 4)}}


def make_variant(kv, device, batch=None):
    case = synth.config5(kv) if batch is None else synth.config5(kv, batch=batch)
    p = synth.make(case, device=device)
    q = p["query"]
    out = torch.empty(tuple(q.shape), dtype=torch.bfloat16, device=device)
    args = ops.make_args(q, p["key_cache"], p["value_cache"], p["block_tables"], p["context_lens"], out,
                         key_scale=p["key_scale"], value_scale=p["value_scale"], q_scale=p["q_scale"],
                         softmax_scale=case.scale_qk(), kernel=KERNEL)
    ws = ops.alloc_workspace(args, device)
    lens = p["context_lens"].cpu().tolist()
    return {"case": case, "p": p, "out": out, "args": args, "ws": ws,
            "bytes": synth.algorithmic_bytes(case, lens), "lens": lens}


def run_ours(a):
    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_attention_decode_02_gb300 import build
    build.build()
    ops.load_library()
    kinds = {"both": [synth.KV_MXFP4, synth.KV_FP8], "mxfp4": [synth.KV_MXFP4],
             "fp8": [synth.KV_FP8]}[a.variant]
    variants = [make_variant(k, dev, a.batch) for k in kinds]
    stream = torch.cuda.current_stream()
    peak, peak_kind = peaks()

    def step(ev=None):
        """One step; with ev, events around each variant's tile kernel."""
        for k, v in enumerate(variants):
            ops.pa_decode_plan(v["args"], v["ws"], stream)
            if ev is not None:
                ev[k][0].record(stream)
            ops.pa_decode(v["args"], v["ws"], stream)
            if ev is not None:
                ev[k][1].record(stream)
            ops.pa_decode_reduce(v["args"], v["ws"], stream)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    for v in variants:
        assert ops.pa_decode_read_status(v["ws"]) == 0, "device status"
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in variants]
           for _ in range(a.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws_n > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        # whole steps, nothing between the launches
        start.record(stream)
        for i in range(a.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        # the same steps again with events around each tile kernel
        for i in range(a.steps):
            step(evs[i])
        torch.cuda.synchronize()
        # each variant's whole call (plan, tile, reduce through pa_decode_run): one call at a
        # time behind a short device-side wait, so that the host's launch time is not counted
        # and no earlier call overlaps it; and the same calls back to back
        call_one, call_b2b = [], []
        for v in variants:
            one = []
            for _ in range(a.steps):
                torch.cuda._sleep(200000)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                ops.pa_decode_run(v["args"], v["ws"], stream)
                e1.record(stream)
                torch.cuda.synchronize()
                one.append(e0.elapsed_time(e1))
            call_one.append(one)
            torch.cuda._sleep(200000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(a.steps):
                ops.pa_decode_run(v["args"], v["ws"], stream)
            e1.record(stream)
            torch.cuda.synchronize()
            call_b2b.append(e0.elapsed_time(e1) / a.steps)
        # the tile kernel launched back to back after one plan (no plan / reduce between)
        b2b = []
        for k, v in enumerate(variants):
            ops.pa_decode_plan(v["args"], v["ws"], stream)
            ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(a.steps)]
            for e0, e1 in ev2:
                e0.record(stream)
                ops.pa_decode(v["args"], v["ws"], stream)
                e1.record(stream)
            torch.cuda.synchronize()
            b2b.append([e0.elapsed_time(e1) for e0, e1 in ev2])
            ops.pa_decode_reduce(v["args"], v["ws"], stream)
    if ws_n > 1:
        torch.distributed.barrier()
    total_ms = start.elapsed_time(end)
    tile_ms = [[evs[i][k][0].elapsed_time(evs[i][k][1]) for i in range(a.steps)]
               for k in range(len(variants))]
    total_ms = replicas.max_over_ranks(total_ms, dev)
    ms_step = total_ms / a.steps
    step_bytes = sum(v["bytes"] for v in variants)
    value = replicas.job_throughput(step_bytes, ms_step, ws_n)

    # end to end through the C ABI with host buffers
    host = []
    for v in variants:
        p = v["p"]
        hq = p["query"].cpu().pin_memory()
        hbt = p["block_tables"].cpu().pin_memory()
        hcl = p["context_lens"].cpu().pin_memory()
        hout = torch.empty(tuple(v["out"].shape), dtype=torch.bfloat16).pin_memory()
        host.append((hq, hbt, hcl, hout))
    h2d = sum(x[0].numel() * x[0].element_size() + x[1].numel() * 4 + x[2].numel() * 4 for x in host)
    d2h = sum(x[3].numel() * 2 for x in host)

    # Two device input / output sets per variant: while step i computes on the compute
    # stream, a copy stream loads step i + 1's query, block tables and context lengths and
    # then reads step i's output back (double buffering, as a serving loop would).
    xs = torch.cuda.Stream(dev)
    sets = []
    for v in variants:
        p = v["p"]
        two = [{"q": p["query"], "bt": p["block_tables"], "cl": p["context_lens"],
                "out": v["out"], "args": v["args"], "ws": v["ws"]}]
        q2, bt2, cl2 = (torch.empty_like(p["query"]), torch.empty_like(p["block_tables"]),
                        torch.empty_like(p["context_lens"]))
        out2 = torch.empty_like(v["out"])
        args2 = ops.make_args(q2, p["key_cache"], p["value_cache"], bt2, cl2, out2,
                              key_scale=p["key_scale"], value_scale=p["value_scale"],
                              q_scale=p["q_scale"], softmax_scale=v["case"].scale_qk(),
                              kernel=KERNEL)
        two.append({"q": q2, "bt": bt2, "cl": cl2, "out": out2, "args": args2,
                    "ws": ops.alloc_workspace(args2, dev)})
        sets.append(two)

    def e2e_run(nsteps):
        """nsteps steps: every one copies its inputs in and its output out."""
        def load(i):  # on the copy stream, after everything it issued before
            with torch.cuda.stream(xs):
                for (hq, hbt, hcl, _), two in zip(host, sets):
                    d = two[i % 2]
                    d["q"].copy_(hq, non_blocking=True)
                    d["bt"].copy_(hbt, non_blocking=True)
                    d["cl"].copy_(hcl, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(xs)
            return ev
        loaded = load(0)
        for i in range(nsteps):
            stream.wait_event(loaded)
            if i + 1 < nsteps:  # set (i+1) % 2 is free: step i-1's output read is queued before
                loaded = load(i + 1)
            for two in sets:
                d = two[i % 2]
                ops.pa_decode_run(d["args"], d["ws"], stream)
            done = torch.cuda.Event()
            done.record(stream)
            xs.wait_event(done)
            with torch.cuda.stream(xs):
                for (_, _, _, hout), two in zip(host, sets):
                    hout.copy_(two[i % 2]["out"], non_blocking=True)
        fin = torch.cuda.Event()
        fin.record(xs)
        stream.wait_event(fin)

    e2e = None
    if not a.no_e2e:
        e2e_run(a.warmup)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        xs.wait_stream(stream)
        e2e_run(a.steps)
        t1.record(stream)
        torch.cuda.synchronize()
        for (_, _, _, hout), v in zip(host, variants):  # the last read-back is the result
            assert torch.equal(hout, v["out"].cpu())
        e2e_ms = replicas.max_over_ranks(t0.elapsed_time(t1) / a.steps, dev)
        e2e_val = replicas.job_throughput(step_bytes, e2e_ms, ws_n)
        e2e = {"value": round(e2e_val, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # per variant: the tile kernel alone and the whole call (plan + tile + reduce), each
    # as µs and as a fraction of the HBM peak; the roofline kernel is the one with the
    # largest share of the step
    var = {}
    for k, v in enumerate(variants):
        tile, call, callb = statistics.median(tile_ms[k]), statistics.median(call_one[k]), call_b2b[k]
        med_b2b = statistics.median(b2b[k])
        frac = lambda ms: round(v["bytes"] / (ms * 1e-3) / 1e9 / peak, 4)
        var[v["case"].name] = {
            "tile_kernel": tile_kernel_name(v["case"]),
            "tile_us": round(tile * 1e3, 2), "tile_frac": frac(tile),
            "tile_us_back_to_back": round(med_b2b * 1e3, 2), "tile_frac_back_to_back": frac(med_b2b),
            "call_us": round(call * 1e3, 2), "call_frac": frac(call),
            "call_us_back_to_back": round(callb * 1e3, 2), "call_frac_back_to_back": frac(callb),
            "share_of_step": round(tile / ms_step, 3), "algorithmic_bytes": v["bytes"]}
    dk = max(range(len(variants)), key=lambda k: statistics.mean(tile_ms[k]))
    dom = variants[dk]
    achieved = dom["bytes"] / (statistics.mean(tile_ms[dk]) * 1e-3) / 1e9
    kname = tile_kernel_name(dom["case"])
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws_n,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "global_batch": 16 * ws_n,
                   "seq_len": "120000-131072", "parallelism": f"replicas x{ws_n}",
                   "l2": "no flush: each call streams more than the 129 MB L2"},
    }
    if a.batch is not None or a.variant != "both":
        line["config"]["note"] = "profiling subset, not the benchmark workload"
    if KERNEL is not None:
        line["config"]["kernel"] = KERNEL
    if not a.no_per_config and a.batch is None and a.variant == "both":
        line["per_config"] = per_config(dev, peak)
    line["gpu_launches"] = 3 * len(variants) * a.steps  # plan, tile, reduce per variant
    line["clocks"] = clk.summary()
    line["e2e"] = e2e
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(variants) if not a.no_cpu_baseline else None
    # last on the line, so that a tail of the output keeps it whole
    line["roofline"] = {"bound": "hbm", "kernel": f"{kname} ({dom['case'].name})",
                        "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_kind,
                        "unit": "GB/s", "frac": round(achieved / peak, 4),
                        "traffic": traffic_from_profile(kname), "variants": var}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        torch.distributed.destroy_process_group()



def _oracle_problem(v, seqs):
    """Oracle view of sequences `seqs` of a bench variant (bytes copied to the host)."""
    from oracle import pa_oracle as orc
    p, case = v["p"], v["case"]
    idx = torch.as_tensor(seqs, dtype=torch.long)
    kv = {synth.KV_MXFP4: orc.KV_MXFP4, synth.KV_FP8: orc.KV_E4M3}[case.kv]
    sk = {synth.SCALE_E8M0: orc.SCALE_E8M0, synth.SCALE_TOKEN: orc.SCALE_TOKEN}[case.scale]
    bt = p["block_tables"].cpu()[idx]
    cl = p["context_lens"].cpu()[idx]
    return orc.Problem(batch=len(seqs), qlen=case.qlen, num_q_heads=case.num_q_heads,
                       num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
                       page_size=case.page_size, num_blocks=p["num_blocks"], kv_format=kv,
                       scale_kind=sk, q_format=orc.Q_BF16, softmax_scale=case.scale_qk(),
                       query=p["query"].cpu()[idx], key_cache=p["key_cache"].cpu(),
                       value_cache=p["value_cache"].cpu(), key_scale=p["key_scale"].cpu(),
                       value_scale=p["value_scale"].cpu(), block_tables=bt, context_lens=cl)


def cpu_baseline(variants, nseq=None):
    """The oracle as it stands, on the host cores, over a bounded sample of the workload."""
    from oracle import pa_oracle as orc
    nseq = nseq or max(1, min(16, orc.max_threads()))
    threads = min(orc.max_threads(), nseq)
    total_bytes, total_s, lens_used = 0, 0.0, 0
    for v in variants:
        seqs = list(range(nseq))
        prob = _oracle_problem(v, seqs)
        t = time.perf_counter()
        prob.decode()
        total_s += time.perf_counter() - t
        lens = [v["lens"][s] for s in seqs]
        # the sample's owned-token KV and scale bytes (its Q, O and table bytes are < 0.01 %)
        total_bytes += sum(lens) * v["case"].num_kv_heads * synth.kv_bytes_per_token(v["case"])
        lens_used += sum(lens)
    return {"value": round(total_bytes / total_s / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"first {nseq} of 16 sequences of each KV variant ({lens_used} tokens), "
                      f"{total_s:.1f} s of fp64 CPU work"}


def run_reference(a):
    """The oracle, timed on the host cores, as the reference arm."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import pa_oracle as orc
    orc.build()
    variants = []
    for kv in (synth.KV_MXFP4, synth.KV_FP8):
        case = synth.config5(kv)
        p = synth.make(case)
        variants.append({"case": case, "p": p, "lens": p["context_lens"].tolist()})
    threads = orc.max_threads()
    nseq = max(1, min(16, threads))  # one (sequence, KV head) unit per host thread
    probs = [_oracle_problem(v, list(range(nseq))) for v in variants]
    sample_bytes = sum(sum(v["lens"][:nseq]) * synth.kv_bytes_per_token(v["case"]) for v in variants)
    for _ in range(a.warmup):
        for pr in probs:
            pr.decode()
    t = time.perf_counter()
    for _ in range(a.steps):
        for pr in probs:
            pr.decode()
    el = (time.perf_counter() - t) / a.steps
    val = sample_bytes / el / 1e9
    threads = min(threads, nseq)
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
            "n_gpus": ws_n, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(el * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD, "global_batch": 16 * ws_n,
                       "seq_len": "120000-131072", "parallelism": f"replicas x{ws_n}",
                       "l2": "no flush: each call streams more than the 129 MB L2"},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"first {nseq} of 16 sequences of each KV variant per step"},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--variant", default="both", choices=["both", "mxfp4", "fp8"],
                    help="KV variants of the long-context workload in a step (profiling: one)")
    ap.add_argument("--batch", type=int, default=None,
                    help="smaller batch for profiling captures (default: the workload's 16)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload µs/call table")
    ap.add_argument("--kernel", default=None, choices=["mma", "tc"],
                    help="decode kernel: the library's choice (default), the mma.sync tile kernel, or the tcgen05 tile kernel")
    ap.add_argument("--kv-write", action="store_true",
                    help="time only the MXFP4 KV-cache write (--steps calls after 3 warm-up) "
                         "and print its line")
    a = ap.parse_args()
    if a.kv_write:
        ops.load_library()
        print(json.dumps(kv_write_config("cuda", peaks()[0], a.steps)))
        return
    global KERNEL
    KERNEL = a.kernel
    if a.warmup < 3 and a.impl == "ours":
        a.warmup = 3
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
