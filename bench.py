#!/usr/bin/env python
"""Benchmark: documents classified per second by trie_tree on one GB300.

Default workload: the Qwen3-4B-shaped final layer (hidden 2,560, 32 q / 8 KV
heads, vocab 151,936) with 256 documents of U{128..1024} tokens and the
10-label support-topic trie ("To Classify, Try a Trie Tree", sec. 2-3); all
inputs seeded and synthetic. One step = one quail_classify_trie_tree call over
all documents (node prologue, tree-masked attention, W_o + RMSNorm, output
head with fused log-sum-exp and child gather, label scoring).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line. The method shards by document with no exchange step,
so N GPUs would be N independent replicas; this benchmark runs one and
refuses --gpus > 1 or a torchrun launch of several ranks. The reference arm
(--impl reference, the CPU oracle) under torchrun runs on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "documents classified/sec at 1 GB300 (trie_tree); % of HBM/tensor roofline"
DEFAULT_WORKLOAD = "qwen3-4b-support10-256docs"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--docs", type=int, default=None, help="override documents per GPU (small profiling cases)")
    p.add_argument("--layers", type=int, default=None, help="override the decoder layers of a multi-layer workload "
                                                            "(small profiling cases)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-other-configs", action="store_true", help="headline workload only")
    p.add_argument("--decode", action="store_true", help="greedy trie_decode instead of trie_tree on a tree workload")
    p.add_argument("--oracle-rate", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--budget", type=float, default=10.0, help=argparse.SUPPRESS)
    return p.parse_args()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    Q = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus = (bus_id or "").lower()
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            c = [x.strip() for x in line.split(",")]
            if len(c) < 10:
                continue
            if self.bus and self.bus[-12:] not in c[1].lower():
                continue
            try:
                sm.append(float(c[2]))
                mx.append(float(c[3]))
                power.append(float(c[4]))
            except ValueError:
                continue
            for n, v in zip(names, c[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ helpers
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def head_kernel_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm.cu", "umma_gemm.cuh", "sm103.cuh"):
        with open(os.path.join(ROOT, "trie_label_scoring_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, rows: int, record: str = "lm_head_gemm_traffic.json"):
    """Per-launch DRAM bytes of a GEMM from a committed ncu summary under
    profiles/, scaled to `rows` if the capture used fewer rows; None once the
    GEMM sources have changed since the capture or for another workload."""
    p = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != head_kernel_hash():
        return None
    if d.get("workload") != workload:
        return None
    return d["dram_bytes_per_launch"] * rows / d["rows"]


def gpu_setup(args) -> None:
    """One process on one GPU. The path shards by document with no exchange
    step (replicas only), and this benchmark runs one replica: a launch on
    several GPUs (torchrun, WORLD_SIZE > 1, or --gpus > 1) is refused."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 or args.gpus != 1:
        sys.stderr.write("bench.py runs on one GPU only: the method shards by document with no exchange step, "
                         "so N GPUs are N independent replicas (trie_label_scoring_gb300.replicas); "
                         f"got --gpus {args.gpus}, WORLD_SIZE {world}\n")
        sys.exit(2)
    import torch
    torch.cuda.set_device(0)


def e2e_entry(n_docs, k_steps, e2e_ms, h2d, d2h, h_in, dev_set) -> dict:
    """The e2e object: docs/s of the end-to-end steps, with the host link's
    own rate beside it (the same pinned tensors copied into one device buffer
    set on a stream of their own, nothing else running; best of three) and
    the docs/s that rate alone would allow."""
    import torch
    st = torch.cuda.Stream()
    best = float("inf")
    for _ in range(3):
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(st)
        with torch.cuda.stream(st):
            for dst, src in zip(dev_set, h_in):
                dst.copy_(src, non_blocking=True)
        e.record(st)
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e))
    link_gbs = h2d / best / 1e6
    value = n_docs * k_steps / (e2e_ms / 1e3)
    link_bound = n_docs / (h2d / (link_gbs * 1e9))
    return {"value": value, "unit": "docs/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": k_steps, "input_buffers": 2, "h2d_link_gbs": link_gbs,
            "h2d_link_bound_docs_s": link_bound, "link_frac": value / link_bound}


def timed_e2e(stream, h_in, dev_sets, call, outs, k_steps) -> float:
    """End-to-end steps through the public API with inputs two buffers deep:
    the host-to-device copy of step i+1's inputs (from pinned host memory, on
    a stream of its own) runs while step i computes on the other device
    buffer; every step's results come back to pinned host memory on the
    compute stream. h_in: pinned host tensors; dev_sets: per buffer, the
    device tensors they are copied to (same order); call(b): the library call
    on buffer b, on `stream`; outs: (device, pinned host) result pairs.
    Returns the ms of k_steps steps, from the start of the first copy to the
    last result read back."""
    import torch
    copy_st = torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in dev_sets]
    free = [torch.cuda.Event() for _ in dev_sets]
    for ev in free:
        ev.record(stream)

    def one(i):
        b = i % len(dev_sets)
        copy_st.wait_event(free[b])  # the step that last read buffer b is done
        with torch.cuda.stream(copy_st):
            for dst, src in zip(dev_sets[b], h_in):
                dst.copy_(src, non_blocking=True)
            ready[b].record(copy_st)
        stream.wait_event(ready[b])
        call(b)
        free[b].record(stream)
        for dev, host in outs:
            host.copy_(dev, non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    copy_st.wait_event(s)
    for i in range(k_steps):
        one(i)
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e)


# ------------------------------------------------------------------ inputs
_MODELS: dict = {}


def model_bits(shape, seed: int = 0) -> dict:
    """The seeded synthetic weights of a layer shape (bf16 bits), drawn once."""
    import synthetic as S
    key = (shape, seed)
    if key not in _MODELS:
        _MODELS[key] = S.make_model(shape, seed)
    return _MODELS[key]


def device_model(shape, seed: int = 0):
    """Those weights on the current GPU as the library's model descriptor."""
    from trie_label_scoring_gb300.torch_inputs import model_from_bits
    return model_from_bits(model_bits(shape, seed), shape)


def oracle_layer(shape, seed: int = 0):
    """The CPU oracle's layer over the same weights (cpu_baseline and the
    reference arm only): fp64, with the head in fp32 beyond a 16,384-token
    vocabulary."""
    import numpy as np

    import oracle.model as OM
    return OM.Layer(model_bits(shape, seed), shape, head_dtype=np.float64 if shape.vocab <= 16384 else np.float32)


def oracle_doc_kv(docs, i: int):
    """Document i's K and V widened exactly to float64 for the oracle."""
    import oracle.model as OM
    k, v = docs.doc_kv(i)
    return OM.bf16_to_f64(k), OM.bf16_to_f64(v)


# ------------------------------------------------------------------ oracle timing
def time_oracle(w, docs, labels, budget_s: float, max_docs: int | None = None) -> dict:
    """The CPU oracle, as it stands, on documents of the same workload until the
    time budget is spent (at least one document)."""
    from oracle import scoring as OS
    from oracle.trie import build_trie
    L = oracle_layer(w.shape)
    L.lm_head()  # widen the head once (model load, not timed)
    t = build_trie(labels.labels, labels.root_token, w.shape.vocab, labels.continuation)
    n, t0 = 0, time.perf_counter()
    limit = max_docs or w.num_docs
    while n < limit:
        dk, dv = oracle_doc_kv(docs, n % w.num_docs)
        OS.trie_tree(L, dk, dv, t)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"docs": n, "seconds": el, "docs_per_s": n / el}


def oracle_rate_one_core(workload: str, docs: int | None, budget_s: float):
    """The oracle's docs/s with BLAS held to one thread: this script re-run in
    --oracle-rate mode in a fresh process (thread counts are read at import)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-rate", "--workload", workload,
           "--budget", str(budget_s)] + (["--docs", str(docs)] if docs else [])
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        line = [l for l in out.stdout.splitlines() if l.startswith("{")][-1]
        return json.loads(line)
    except (subprocess.SubprocessError, IndexError, ValueError, OSError):
        return None


def run_oracle_rate(args):
    """--oracle-rate: the oracle alone on a bounded sample; one JSON line."""
    import synthetic as S
    w = S.WORKLOADS[args.workload]
    if args.docs:
        w = S.with_docs(w, args.docs)
    r = time_oracle(w, S.make_docs(w, 0), S.make_labels(w, 0), budget_s=args.budget)
    print(json.dumps({"value": r["docs_per_s"], "unit": "docs/s", "cores": 1, "docs": r["docs"],
                      "seconds": r["seconds"], "threads_env": os.environ.get("OPENBLAS_NUM_THREADS")}), flush=True)


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return
    import synthetic as S
    from oracle import scoring as OS
    from oracle.trie import build_trie
    if args.workload in S.ML_WORKLOADS:
        run_reference_ml(args, world)
        return
    if args.workload in S.SHORTLIST_WORKLOADS:
        run_reference_shortlist(args, world)
        return
    w = S.WORKLOADS[args.workload]
    if args.docs:
        w = S.with_docs(w, args.docs)
    labels = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    L = oracle_layer(w.shape)
    L.lm_head()
    t = build_trie(labels.labels, labels.root_token, w.shape.vocab, labels.continuation)
    steps = args.steps if args.steps is not None else 10

    def step(i):
        dk, dv = oracle_doc_kv(docs, i % w.num_docs)
        OS.trie_tree(L, dk, dv, t)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = steps / el
    sample = f"1 document of {w.name} per step (oracle trie_tree: fp64 layer, fp32 head GEMV, fp64 LSE)"
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "docs/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * el / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "docs_per_step": 1},
        "cpu_baseline": {"value": value, "unit": "docs/s", "cores": cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "docs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_reference_ml(args, world):
    """The multi-layer oracle on one document per step (see time_oracle_ml)."""
    import synthetic as S
    mw = S.ML_WORKLOADS[args.workload]
    base = S.with_docs(mw.base, args.docs) if args.docs else mw.base
    bits = S.make_model_ml(base.shape, 2, mw.intermediate, 0)
    docs_ml = S.make_docs_ml(base, 2, 0)
    labels = S.make_labels(base, 0)
    steps = args.steps if args.steps is not None else 1
    rates = [time_oracle_ml(mw, base, bits, docs_ml, labels, budget_s=60.0) for _ in range(steps)]
    value = statistics.mean(r["docs_per_s"] for r in rates)
    sample = (f"document 0 of {base.name} through the first 1 and 2 layers per step; time per document "
              f"extrapolated to {mw.n_layers} layers")
    out = {
        "impl": "reference", "metric": f"documents classified/sec at 1 GB300 (trie_tree through {mw.n_layers} "
                                       f"decoder layers)",
        "value": value, "unit": "docs/s", "n_gpus": world, "steps": steps, "warmup": 0,
        "ms_per_step": 1e3 / value, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)", "config": {"workload": mw.name, "docs_per_step": 1},
        "cpu_baseline": {"value": value, "unit": "docs/s", "cores": cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "docs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_reference_shortlist(args, world):
    """The shortlist oracle on one document per step."""
    import synthetic as S
    from oracle import shortlist as OSL
    from oracle.trie import build_trie
    sw = S.SHORTLIST_WORKLOADS[args.workload]
    w = S.with_docs(sw.base, args.docs) if args.docs else sw.base
    labels = S.make_labels(w, 0)
    K = len(labels.labels)
    G = sw.groups or OSL.default_groups(K)
    names = S.make_group_names(0, G, 1, w.shape.vocab)
    rw = OSL.rewrite_grouped(labels.labels, names, OSL.group_labels(labels.labels, G))
    t = build_trie(rw, labels.root_token, w.shape.vocab)
    docs = S.make_docs(w, 0)
    L = oracle_layer(w.shape)
    L.lm_head()
    steps = args.steps if args.steps is not None else 3

    def step(i):
        dk, dv = oracle_doc_kv(docs, i % w.num_docs)
        OSL.shortlist(L, dk, dv, t, 1, sw.beam)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = steps / el
    out = {
        "impl": "reference", "metric": "documents classified/sec at 1 GB300 (shortlisted trie_tree over grouped "
                                       "labels)",
        "value": value, "unit": "docs/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)", "config": {"workload": sw.name, "docs_per_step": 1},
        "cpu_baseline": {"value": value, "unit": "docs/s", "cores": cores(), "kind": "oracle",
                         "sample": f"1 document of {w.name} per step (oracle shortlist, {G} groups, beam {sw.beam})"},
        "e2e": {"value": value, "unit": "docs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import numpy as np
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import bf16_tensor, kv_from_docs

    Q.build()
    w = S.WORKLOADS[args.workload]
    if args.docs:
        w = S.with_docs(w, args.docs)
    model = device_model(w.shape, 0)
    labels = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    tb0 = time.perf_counter()
    trie = Q.Trie(labels.labels, labels.root_token, w.shape.vocab, labels.continuation)
    trie_build_ms = 1e3 * (time.perf_counter() - tb0)  # host build, outside the timed region
    trie.upload()
    N, M, a = w.num_docs, len(labels.labels), trie.n_eval
    view = trie.view()
    n_children = np.diff(view["child_offsets"])
    trie_stats = {"nodes": int(view["n_nodes"]), "evaluated": int(a), "build_ms": trie_build_ms,
                  "depth_histogram": np.bincount(view["depth"]).tolist(),
                  "mean_branching": float(n_children[n_children > 0].mean()),
                  "branching_nodes": int(view["is_branching"].sum())}
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_TREE), dtype=torch.uint8,
                     device="cuda")
    lsc = torch.empty((N, M), device="cuda")
    prob = torch.empty((N, M), device="cuda")
    am = torch.empty((N,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.classify_trie_tree(model, kv, trie, N, ws, lsc, prob, am, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    Q.device_status()
    launches_per_step = Q.launch_count()  # kernels one call launches, counted by the library
    # choose K: about 2 s of device time unless given
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    step()
    t1.record(stream)
    t1.synchronize()
    est_ms = t0.elapsed_time(t1)
    steps = args.steps if args.steps is not None else int(min(5000, max(20, 2000.0 / max(est_ms, 1e-3))))

    # stage events for every step (10 per step: begin/end of the 5 stages); the
    # head GEMM's pair (stage 3) gives the roofline kernel's own duration
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(steps)]
    for evs in stage_ev:  # torch creates the CUDA event on first record; the library re-records it
        for e in evs:
            e.record(stream)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(0).pci_bus_id
    except Exception:
        pass
    clocks = ClockSampler(str(bus) if bus is not None else None)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # Inside the timed loop only the head GEMM's pair of events is recorded (the
    # roofline kernel); an event between two kernels keeps the second from
    # launching while the first drains, so the other stage boundaries are timed
    # in a separate loop after this one.
    hs = Q.STAGES.index("head")
    start.record(stream)
    for k in range(steps):
        Q.set_stage_events([None] * (2 * hs) + stage_ev[k][2 * hs: 2 * hs + 2])
        step()
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    Q.set_stage_events(None)
    Q.device_status()
    elapsed_ms = start.elapsed_time(end)
    head_ms = statistics.mean(ev[2 * hs].elapsed_time(ev[2 * hs + 1]) for ev in stage_ev)
    ms_per_step = elapsed_ms / steps
    value = N * steps / (elapsed_ms / 1e3)
    # stage breakdown (every boundary marked), after the timed region
    n_bd = min(steps, 50)
    bd_ev = stage_ev[:n_bd]
    torch.cuda.synchronize()
    for k in range(n_bd):
        Q.set_stage_events(bd_ev[k])
        step()
    torch.cuda.synchronize()
    Q.set_stage_events(None)
    stages_ms = {name: statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for ev in bd_ev)
                 for i, name in enumerate(Q.STAGES)}

    # ---- e2e: host buffers through the C ABI, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        hk = bf16_tensor(docs.k_pool, "cpu").pin_memory()
        hv = bf16_tensor(docs.v_pool, "cpu").pin_memory()
        hpt = torch.from_numpy(docs.page_table).pin_memory()
        hdl = torch.from_numpy(docs.doc_len).pin_memory()
        o_ls = torch.empty((N, M)).pin_memory()
        o_pr = torch.empty((N, M)).pin_memory()
        o_am = torch.empty((N,), dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hpt, hdl))
        d2h = sum(t.numel() * t.element_size() for t in (o_ls, o_pr, o_am))

        kvs = [kv, kv_from_docs(docs)]  # two device KV buffers: copy one while the other computes

        def e2e_call(b):
            Q.classify_trie_tree(model, kvs[b], trie, N, ws, lsc, prob, am, stream)

        k_e2e = max(3, min(steps, int(3000.0 / max(est_ms + 3.0, 1e-3))))
        e2e_ms = timed_e2e(stream, [hk, hv, hpt, hdl], [list(x.tensors) for x in kvs], e2e_call,
                           [(lsc, o_ls), (prob, o_pr), (am, o_am)], k_e2e)
        e2e = e2e_entry(N, k_e2e, e2e_ms, h2d, d2h, [hk, hv, hpt, hdl], list(kvs[1].tensors))

    # ---- roofline of the dominant kernel (the output-head GEMM)
    peaks = measured_peaks()
    rows = N * a
    d, V = w.shape.hidden, w.shape.vocab
    flops = 2.0 * d * V * rows
    achieved = flops / (head_ms / 1e3) / 1e12
    traffic = recorded_traffic(w.name, rows)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": traffic, "kernel": "umma_gemm_kernel<EpiHead>",
                "head_ms": head_ms, "peak_kind": f"bf16 burst ({peaks['source']})",
                "frac_sustained": (achieved / peaks["bf16_tflops_sustained"]
                                   if peaks.get("bf16_tflops_sustained") else None),
                "frac_spec": achieved / SPEC_BF16_TFLOPS}
    # ---- path roofline: max(KV bytes / HBM, head FLOPs / tensor peak)
    kv_bytes = float(docs.doc_len.sum()) * w.shape.n_kv_heads * w.shape.head_dim * 2 * 2
    t_kv = kv_bytes / (peaks["hbm_gbs"] * 1e9)
    t_head = flops / (peaks["bf16_tflops"] * 1e12)
    t_star = max(t_kv, t_head)
    path = {"t_kv_us": t_kv * 1e6, "t_head_us": t_head * 1e6, "t_star_us": t_star * 1e6,
            "ms_per_step": ms_per_step, "frac": t_star * 1e3 / ms_per_step}

    # ---- CPU baseline: the oracle on a bounded sample,
    # on all host cores and, in a subprocess with single-threaded BLAS, on one
    cpu = None
    if not args.no_cpu_baseline:
        r = time_oracle(w, docs, labels, budget_s=15.0)
        cpu = {"value": r["docs_per_s"], "unit": "docs/s", "cores": cores(), "kind": "oracle",
               "sample": f"first {r['docs']} documents of {w.name} ({r['seconds']:.1f} s); numpy BLAS threads "
                         f"default to all {cores()} cores"}
        one = oracle_rate_one_core(w.name, args.docs, budget_s=10.0)
        if one is not None:
            cpu["one_core"] = one

    # ---- the other workloads (larger label sets, long documents, letters, decode), after the headline, same steps and warm-up
    others = None
    if w.name == DEFAULT_WORKLOAD and not args.no_other_configs:
        others = measure_other_configs(model, args.steps if args.steps is not None else 20, max(args.warmup, 3))

    out = {
        "metric": METRIC, "value": value, "unit": "docs/s", "n_gpus": 1, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": w.name, "docs_per_gpu": N, "labels": M, "eval_positions_per_doc": a,
                   "trie_nodes": trie.n_nodes, "trie": trie_stats, "hidden": d, "vocab": V,
                   "q_heads": w.shape.n_q_heads,
                   "kv_heads": w.shape.n_kv_heads, "doc_tokens_per_gpu": int(docs.doc_len.sum()),
                   "l2": "inputs larger than L2 (doc KV %.2f GB + output head %.2f GB per step)" % (
                       kv_bytes / 1e9, 2.0 * d * V / 1e9),
                   "parallelism": "one replica (documents shard across GPUs with no collective)"},
        "roofline": roofline, "path_roofline": path, "stages_ms": stages_ms, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * steps, "clocks": clk, "other_configs": others,
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ the other configurations
# Measured in the same process as the headline, with the same step and
# warm-up counts: the larger label sets, the long documents and the two
# variants that fall out of the same kernels.
OTHER_CONFIGS = (
    ("tree255-64x2048", "qwen3-4b-tree255-64x2048", "trie_tree"),
    ("letters255-64x2048", "qwen3-4b-letters255-64x2048", "letters"),
    ("tree20-32x8192", "qwen3-4b-tree20-32x8192", "trie_tree"),
    ("tree20-32x8192 decode", "qwen3-4b-tree20-32x8192", "decode"),
    ("tree5000-16x1024", "qwen3-4b-tree5000-16x1024", "trie_tree"),
)
SPEC_BF16_TFLOPS = 2250.0  # nominal dense bf16 of one GB300 (context next to the measured peaks)


def _stage_breakdown(Q, step, n: int) -> dict:
    """Mean stage spans over n calls, every boundary marked (after a timed loop)."""
    import torch
    stream = torch.cuda.current_stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(Q.STAGES))] for _ in range(n)]
    for e in evs:
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for e in evs:
        Q.set_stage_events(e)
        step()
    torch.cuda.synchronize()
    Q.set_stage_events(None)
    return {name: statistics.mean(e[2 * i].elapsed_time(e[2 * i + 1]) for e in evs)
            for i, name in enumerate(Q.STAGES)}


def _leg_trie_tree(Q, w, model, docs, labels, steps: int, warmup: int) -> dict:
    import torch

    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    kv = kv_from_docs(docs)
    trie = Q.Trie(labels.labels, labels.root_token, w.shape.vocab, labels.continuation)
    trie.upload()
    N, M, a = w.num_docs, len(labels.labels), trie.n_eval
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_TREE), dtype=torch.uint8,
                     device="cuda")
    lsc = torch.empty((N, M), device="cuda")
    prob = torch.empty((N, M), device="cuda")
    am = torch.empty((N,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.classify_trie_tree(model, kv, trie, N, ws, lsc, prob, am, stream)

    for _ in range(warmup):
        step()
    Q.device_status()
    launches = Q.launch_count()
    hs = Q.STAGES.index("head")
    elapsed_ms, stage_ev, clk = _timed_loop(stream, steps, step, 2 * len(Q.STAGES), keep=(2 * hs, 2 * hs + 1))
    head_ms = statistics.mean(ev[2 * hs].elapsed_time(ev[2 * hs + 1]) for ev in stage_ev)
    stages = _stage_breakdown(Q, step, min(steps, 10))
    peaks = measured_peaks()
    ms = elapsed_ms / steps
    d, V = w.shape.hidden, w.shape.vocab
    flops = 2.0 * d * V * N * a
    kv_bytes = float(docs.doc_len.sum()) * w.shape.n_kv_heads * w.shape.head_dim * 2 * 2
    t_kv = kv_bytes / (peaks["hbm_gbs"] * 1e9)
    t_head = flops / (peaks["bf16_tflops"] * 1e12)
    head_tf = flops / (head_ms / 1e3) / 1e12
    view = trie.view()
    out = {"workload": w.name, "kind": "trie_tree", "docs": N, "labels": M, "eval_positions_per_doc": a,
           "trie_nodes": int(view["n_nodes"]), "trie_max_depth": int(view["depth"].max()),
           "ms_per_step": ms, "docs_per_s": N * steps / (elapsed_ms / 1e3),
           "path_roofline": {"t_kv_us": t_kv * 1e6, "t_head_us": t_head * 1e6,
                             "frac": max(t_kv, t_head) * 1e3 / ms},
           "head": {"ms": head_ms, "achieved_tflops": head_tf, "frac": head_tf / peaks["bf16_tflops"],
                    "frac_sustained": (head_tf / peaks["bf16_tflops_sustained"]
                                       if peaks.get("bf16_tflops_sustained") else None),
                    "frac_spec": head_tf / SPEC_BF16_TFLOPS},
           "stages_ms": stages, "gpu_launches": launches * steps, "clocks": clk}
    del kv, ws
    return out


def _leg_letters(Q, w, model, docs, labels, steps: int, warmup: int) -> dict:
    import torch

    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    kv = kv_from_docs(docs)
    tokens = [l[0] for l in labels.labels]
    N, M = w.num_docs, len(tokens)
    ws = torch.empty(Q.workspace_size(model, None, M, N, docs.max_doc_len, Q.MODE_LETTERS), dtype=torch.uint8,
                     device="cuda")
    lp = torch.empty((N, M), device="cuda")
    pr = torch.empty((N, M), device="cuda")
    am = torch.empty((N,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.classify_letters(model, kv, tokens, labels.root_token, N, ws, lp, pr, am, stream)

    for _ in range(warmup):
        step()
    Q.device_status()
    launches = Q.launch_count()
    ai = Q.STAGES.index("attention")
    elapsed_ms, stage_ev, clk = _timed_loop(stream, steps, step, 2 * len(Q.STAGES), keep=(2 * ai, 2 * ai + 1))
    att_ms = statistics.mean(ev[2 * ai].elapsed_time(ev[2 * ai + 1]) for ev in stage_ev)
    peaks = measured_peaks()
    ms = elapsed_ms / steps
    kv_bytes = float(docs.doc_len.sum()) * w.shape.n_kv_heads * w.shape.head_dim * 2 * 2
    t_kv = kv_bytes / (peaks["hbm_gbs"] * 1e9)
    out = {"workload": w.name, "kind": "letters", "docs": N, "letters": M, "ms_per_step": ms,
           "docs_per_s": N * steps / (elapsed_ms / 1e3),
           "path_roofline": {"t_kv_us": t_kv * 1e6, "frac": t_kv * 1e3 / ms},
           "attention": {"ms": att_ms, "achieved_gbs": kv_bytes / (att_ms / 1e3) / 1e9,
                         "frac": kv_bytes / (att_ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
           "gpu_launches": launches * steps, "clocks": clk}
    del kv, ws
    return out


def _leg_decode(Q, w, model, docs, labels, steps: int, warmup: int) -> dict:
    import torch

    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    kv = kv_from_docs(docs)
    trie = Q.Trie(labels.labels, labels.root_token, w.shape.vocab, labels.continuation)
    trie.upload()
    N = w.num_docs
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_DECODE), dtype=torch.uint8,
                     device="cuda")
    cur = torch.zeros(N, dtype=torch.int32, device="cuda")
    lab = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    act = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    n_steps = 0
    while True:  # how many decode steps this batch takes
        Q.classify_trie_decode_step(model, kv, trie, N, cur, lab, act, ws, None, stream)
        n_steps += 1
        if int(act.item()) == 0 or n_steps >= 64:
            break
    launches = Q.launch_count()

    def decode():
        cur.zero_()
        lab.fill_(-1)
        for _ in range(n_steps):
            Q.classify_trie_decode_step(model, kv, trie, N, cur, lab, act, ws, None, stream)

    for _ in range(warmup):
        decode()
    Q.device_status()
    elapsed_ms, _, clk = _timed_loop(stream, steps, decode)
    ms = elapsed_ms / steps
    out = {"workload": w.name, "kind": "trie_decode", "docs": N, "labels": len(labels.labels),
           "decode_steps": n_steps, "ms_per_batch": ms, "docs_per_s": N * steps / (elapsed_ms / 1e3),
           "gpu_launches": launches * n_steps * steps, "clocks": clk,
           "note": "one step = the whole greedy decode of the batch; reported, not graded"}
    del kv, ws
    return out


def measure_other_configs(model, steps: int, warmup: int) -> dict:
    """Every other configuration of the method on the same GPU, one after the
    other; documents of the same shape are generated once."""
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    legs = {"trie_tree": _leg_trie_tree, "letters": _leg_letters, "decode": _leg_decode}
    docs_cache: dict = {}
    out = {}
    for label, name, kind in OTHER_CONFIGS:
        w = S.WORKLOADS[name]
        key = (w.shape, w.num_docs, w.doc_len)
        if key not in docs_cache:
            docs_cache.clear()
            docs_cache[key] = S.make_docs(w, 0)
        out[label] = legs[kind](Q, w, model, docs_cache[key], S.make_labels(w, 0), steps, warmup)
        torch.cuda.empty_cache()
    return out


def run_join(args):
    """AI.IF over joined pairs: every anchor document against every partner
    (quail_join_if). One step = one call over all anchors; metric = pairs/s."""
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs

    Q.build()
    w = S.WORKLOADS[args.workload]
    if args.docs:
        w = S.with_docs(w, args.docs)
    model = device_model(w.shape, 0)
    partners = S.make_labels(w, 0)
    yes, no = S.make_answers(0, w.shape.vocab)
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    trie = Q.Trie(partners.labels, partners.root_token, w.shape.vocab, all_nodes=True)
    trie.upload()
    N, M = w.num_docs, len(partners.labels)
    ws = torch.empty(Q.workspace_size(model, trie, len(yes) + len(no), N, docs.max_doc_len, Q.MODE_JOIN_IF),
                     dtype=torch.uint8, device="cuda")
    p_true = torch.empty((N, M), device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.join_if(model, kv, trie, N, yes, no, ws, p_true, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    Q.device_status()
    launches_per_step = Q.launch_count()
    steps = args.steps if args.steps is not None else 50
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(steps)]
    for evs in stage_ev:
        for e in evs:
            e.record(stream)
    clocks = ClockSampler(str(torch.cuda.get_device_properties(0).pci_bus_id))
    clocks.start()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ai = Q.STAGES.index("attention")  # only the roofline kernel's events inside the timed loop
    start.record(stream)
    for k in range(steps):
        Q.set_stage_events([None] * (2 * ai) + stage_ev[k][2 * ai: 2 * ai + 2])
        step()
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    Q.set_stage_events(None)
    Q.device_status()
    elapsed_ms = start.elapsed_time(end)
    attention_ms = statistics.mean(ev[2 * ai].elapsed_time(ev[2 * ai + 1]) for ev in stage_ev)
    bd_ev = stage_ev[:min(steps, 20)]  # stage breakdown, after the timed region
    for evs in bd_ev:
        Q.set_stage_events(evs)
        step()
    torch.cuda.synchronize()
    Q.set_stage_events(None)
    stages_ms = {name: statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for ev in bd_ev)
                 for i, name in enumerate(Q.STAGES[:4])}
    ms_per_step = elapsed_ms / steps
    pairs = N * M
    # dominant kernel: the doc-part attention (tcgen05, G * M query rows per KV head);
    # its algorithmic work is 4 * 128 FLOP per (query row, anchor key)
    G = w.shape.n_q_heads // w.shape.n_kv_heads
    keys = float(docs.doc_len.sum())
    attn_flops = 4.0 * 128 * keys * w.shape.n_kv_heads * G * M
    peaks = measured_peaks()
    achieved = attn_flops / (attention_ms / 1e3) / 1e12
    kv_bytes = keys * w.shape.n_kv_heads * 128 * 2 * 2
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": None, "kernel": "attn_doc_tc_kernel",
                "attention_ms": attention_ms, "peak_kind": f"bf16 burst ({peaks['source']})",
                "note": "FLOPs counted once per query row (the hi/lo splits double the issued work)"}
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import join as J
        L = oracle_layer(w.shape, 0)
        t0 = time.time()
        done = 0
        dk, dv = oracle_doc_kv(docs, 0)
        while done < M and time.time() - t0 < 15.0:
            J.join_if(L, dk, dv, partners.root_token, [partners.labels[done]], yes, no)
            done += 1
        sec = time.time() - t0
        cpu = {"value": done / sec, "unit": "pairs/s", "cores": cores(), "kind": "oracle",
               "sample": f"anchor 0 with its first {done} partners ({sec:.1f} s)"}
    out = {
        "metric": "joined pairs scored/sec at 1 GB300 (AI.IF, TRUE/FALSE head)",
        "value": pairs * steps / (elapsed_ms / 1e3), "unit": "pairs/s", "n_gpus": 1,
        "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": w.name, "anchors_per_gpu": N, "partners": M, "partner_trie_nodes": trie.n_nodes,
                   "answer_spellings": len(yes) + len(no), "anchor_tokens_per_gpu": int(keys),
                   "l2": "anchor KV %.2f GB per step" % (kv_bytes / 1e9),
                   "parallelism": "one replica (anchors shard across GPUs with no collective)"},
        "roofline": roofline, "stages_ms": stages_ms, "cpu_baseline": cpu, "e2e": None,
        "gpu_launches": launches_per_step * steps, "clocks": clk,
    }
    print(json.dumps(out), flush=True)


def time_oracle_ml(mw, base, bits, docs_ml, labels, budget_s: float) -> dict:
    """The multi-layer oracle, as it stands, on document 0 through the first
    one and the first two layers of the stack; the full stack's time per
    document is extrapolated as t1 + (n_layers - 1) * (t2 - t1)."""
    import numpy as np

    from oracle import multilayer as ML
    from oracle.trie import build_trie
    d0, ks, vs = docs_ml
    n = int(d0.doc_len[0])
    pages = d0.page_table[0, : (n + 15) // 16]

    def kv(l):
        import oracle.model as OM
        k = ks[l][pages].transpose(0, 2, 1, 3).reshape(-1, ks[l].shape[1], ks[l].shape[3])[:n]
        v = vs[l][pages].transpose(0, 2, 1, 3).reshape(-1, vs[l].shape[1], vs[l].shape[3])[:n]
        return OM.bf16_to_f64(k), OM.bf16_to_f64(v)

    t = build_trie(labels.labels, labels.root_token, base.shape.vocab, labels.continuation)
    head = np.float64 if base.shape.vocab <= 16384 else np.float32
    times = {}
    t_all = time.perf_counter()
    for L in (1, 2):
        md = ML.ModelML(dict(bits, layers=bits["layers"][:L]), base.shape, head_dtype=head)
        md.lm_head()  # widen the head once (model load, not timed)
        doc_kv = [kv(l) for l in range(L)]
        t0 = time.perf_counter()
        ML.trie_tree(md, doc_kv, t)
        times[L] = time.perf_counter() - t0
        if time.perf_counter() - t_all > budget_s:
            break
    t1 = times[1]
    t2 = times.get(2, 2 * t1)
    per_layer = max(t2 - t1, t1 / 2)
    t_doc = t1 + (mw.n_layers - 1) * per_layer
    return {"docs_per_s": 1.0 / t_doc, "t1": t1, "t2": t2, "t_doc": t_doc}


def run_ml(args):
    """trie_tree through the whole decoder stack (quail_classify_trie_tree_ml).
    One step = one call over all documents; metric = documents/s."""
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_ml_from_docs, model_ml_from_bits

    Q.build()
    mw = S.ML_WORKLOADS[args.workload]
    if args.layers:
        mw = S.MLWorkload(f"{mw.name}[{args.layers} layers]", mw.base, args.layers, mw.intermediate)
    base = S.with_docs(mw.base, args.docs) if args.docs else mw.base
    L, I = mw.n_layers, mw.intermediate
    sh = base.shape
    bits = S.make_model_ml(sh, L, I, 0)
    model = model_ml_from_bits(bits, sh, I)
    labels = S.make_labels(base, 0)
    docs_ml = S.make_docs_ml(base, L, 0)
    d0 = docs_ml[0]
    kv = kv_ml_from_docs(*docs_ml)
    trie = Q.Trie(labels.labels, labels.root_token, sh.vocab, labels.continuation)
    trie.upload()
    N, M, a = base.num_docs, len(labels.labels), trie.n_eval
    rows = N * a
    ws = torch.empty(Q.workspace_size_ml(model, trie, N, d0.max_doc_len), dtype=torch.uint8, device="cuda")
    lsc = torch.empty((N, M), device="cuda")
    prob = torch.empty((N, M), device="cuda")
    am = torch.empty((N,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.classify_trie_tree_ml(model, kv, trie, N, ws, lsc, prob, am, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    Q.device_status()
    launches_per_step = Q.launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    step()
    t1.record(stream)
    t1.synchronize()
    est_ms = t0.elapsed_time(t1)
    steps = args.steps if args.steps is not None else int(min(400, max(20, 2000.0 / max(est_ms, 1e-3))))
    n_ev = 2 * (len(Q.STAGES) + len(Q.LAYER_SPANS) * L)
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    for evs in stage_ev:
        for e in evs:
            e.record(stream)
    # inside the timed loop only the gate|up spans (the roofline kernel) are
    # marked, since an event between two kernels keeps the second from
    # launching while the first drains; the full breakdown is a separate loop
    s0, nsp, gu = len(Q.STAGES), len(Q.LAYER_SPANS), Q.LAYER_SPANS.index("gate_up")
    gu_idx = [2 * (s0 + l * nsp + gu) + j for l in range(L) for j in (0, 1)]

    def timed_events(evs):
        sel = [None] * len(evs)
        for i in gu_idx:
            sel[i] = evs[i]
        return sel
    clocks = ClockSampler(str(torch.cuda.get_device_properties(0).pci_bus_id))
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        Q.set_stage_events(timed_events(stage_ev[k]))
        step()
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    Q.set_stage_events(None)
    Q.device_status()
    elapsed_ms = start.elapsed_time(end)
    ms_per_step = elapsed_ms / steps
    value = N * steps / (elapsed_ms / 1e3)
    gate_up_ms = statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in stage_ev for i in gu_idx[::2])
    # breakdown with every stage and span marked, after the timed region
    bd_ev = stage_ev[:min(steps, 10)]
    torch.cuda.synchronize()
    for evs in bd_ev:
        Q.set_stage_events(evs)
        step()
    torch.cuda.synchronize()
    Q.set_stage_events(None)
    stages_ms = {name: statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for ev in bd_ev)
                 for i, name in enumerate(Q.STAGES) if name != "attention" and name != "wo_norm"}
    span_ms = {}
    for j, name in enumerate(Q.LAYER_SPANS):
        span_ms[name] = statistics.mean(ev[2 * (s0 + l * nsp + j)].elapsed_time(ev[2 * (s0 + l * nsp + j) + 1])
                                        for ev in bd_ev for l in range(L))

    # ---- e2e: every layer's document KV from pinned host memory, results back
    e2e = None
    if not args.no_e2e:
        from trie_label_scoring_gb300.torch_inputs import bf16_tensor
        _, ks, vs = docs_ml
        hks = [bf16_tensor(k, "cpu").pin_memory() for k in ks]
        hvs = [bf16_tensor(v, "cpu").pin_memory() for v in vs]
        hpt = torch.from_numpy(d0.page_table).pin_memory()
        hdl = torch.from_numpy(d0.doc_len).pin_memory()
        o_ls = torch.empty((N, M)).pin_memory()
        o_pr = torch.empty((N, M)).pin_memory()
        o_am = torch.empty((N,), dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in hks + hvs + [hpt, hdl])
        d2h = sum(t.numel() * t.element_size() for t in (o_ls, o_pr, o_am))

        kvs = [kv, kv_ml_from_docs(*docs_ml)]  # two device KV buffers: copy one while the other computes

        def e2e_call(b):
            Q.classify_trie_tree_ml(model, kvs[b], trie, N, ws, lsc, prob, am, stream)

        def flat(k):
            kd, vd, pt, dl = k.tensors
            return list(kd) + list(vd) + [pt, dl]

        k_e2e = max(3, min(steps, 10))
        e2e_ms = timed_e2e(stream, hks + hvs + [hpt, hdl], [flat(x) for x in kvs], e2e_call,
                           [(lsc, o_ls), (prob, o_pr), (am, o_am)], k_e2e)
        e2e = e2e_entry(N, k_e2e, e2e_ms, h2d, d2h, hks + hvs + [hpt, hdl], flat(kvs[1]))

    # ---- roofline of the dominant kernel: the gate|up GEMM of a layer, with
    # SiLU(gate) * up fused into its epilogue (output: the two-term bf16 split
    # of the activation, 4 bytes per element)
    peaks = measured_peaks()
    d, V = sh.hidden, sh.vocab
    gu_bytes = 2.0 * d * 2 * I + 2.0 * rows * d + 4.0 * rows * I
    gu_flops = 2.0 * rows * d * 2 * I
    t_gu = gate_up_ms / 1e3
    if gu_bytes / (peaks["hbm_gbs"] * 1e9) >= gu_flops / (peaks["bf16_tflops"] * 1e12):
        achieved = gu_bytes / t_gu / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "peak_kind": f"HBM copy ({peaks['source']})"}
    else:
        achieved = gu_flops / t_gu / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"], "peak_kind": f"bf16 burst ({peaks['source']})"}
    roofline.update({"traffic": recorded_traffic(mw.name, rows, "gate_up_gemm_traffic.json"),
                     "kernel": "umma_gemm_kernel<EpiSwiGLU> (gate|up, split A, SwiGLU epilogue)",
                     "gate_up_ms": gate_up_ms, "algorithmic_bytes": gu_bytes,
                     "algorithmic_flops": gu_flops,
                     "issued_tflops": 2 * gu_flops / t_gu / 1e12,
                     "note": "A is a two-term bf16 split, so the issued MMA work is twice the algorithmic FLOPs"})
    # ---- path roofline: all weight and document-KV bytes vs all GEMM FLOPs
    hq, hkv, hd = sh.n_q_heads, sh.n_kv_heads, sh.head_dim
    layer_params = d * (hq + 2 * hkv) * hd + hq * hd * d + 3 * d * I
    keys = float(d0.doc_len.sum())
    kv_bytes = keys * hkv * hd * 2 * 2 * L
    path_bytes = 2.0 * layer_params * L + kv_bytes + 2.0 * d * V
    path_flops = 2.0 * rows * (layer_params * L + d * V) + 4.0 * hd * keys * hq * a * L
    t_b = path_bytes / (peaks["hbm_gbs"] * 1e9)
    t_f = path_flops / (peaks["bf16_tflops"] * 1e12)
    path = {"t_bytes_us": t_b * 1e6, "t_flops_us": t_f * 1e6, "t_star_us": max(t_b, t_f) * 1e6,
            "ms_per_step": ms_per_step, "frac": max(t_b, t_f) * 1e3 / ms_per_step,
            "bytes_per_step": path_bytes, "flops_per_step": path_flops}

    cpu = None
    if not args.no_cpu_baseline:
        r = time_oracle_ml(mw, base, bits, docs_ml, labels, budget_s=60.0)
        cpu = {"value": r["docs_per_s"], "unit": "docs/s", "cores": cores(), "kind": "oracle",
               "sample": f"document 0 of {base.name} through the first 1 and 2 layers ({r['t1']:.1f} s, "
                         f"{r['t2']:.1f} s); per-document time extrapolated to {L} layers = {r['t_doc']:.1f} s"}
    out = {
        "metric": f"documents classified/sec at 1 GB300 (trie_tree through {L} decoder layers)",
        "value": value, "unit": "docs/s", "n_gpus": 1, "steps": steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": mw.name, "docs_per_gpu": N, "labels": M, "eval_positions_per_doc": a,
                   "rows": rows, "layers": L, "intermediate": I, "hidden": d, "vocab": V,
                   "doc_tokens_per_gpu": int(keys),
                   "l2": "inputs larger than L2 (weights %.2f GB + document KV %.2f GB per step)" % (
                       2.0 * layer_params * L / 1e9, kv_bytes / 1e9),
                   "parallelism": "one replica (documents shard across GPUs with no collective)"},
        "roofline": roofline, "path_roofline": path, "stages_ms": stages_ms, "layer_spans_ms": span_ms,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * steps, "clocks": clk,
    }
    print(json.dumps(out), flush=True)


def _group_rows(view, D: int) -> dict:
    """Rows of each group of a shortlist plan at cut depth D: the evaluated
    ancestors of the group's depth-D node plus the evaluated nodes of its
    subtree (node order = group order)."""
    import numpy as np
    depth, parent, sub, ev = view["depth"], view["parent"], view["subtree_size"], view["eval_index_of_node"] >= 0
    nodes = np.nonzero(depth == D)[0]
    cum = np.concatenate([[0], np.cumsum(ev)])
    rows = []
    for c in nodes:
        up, u = 0, int(parent[c])
        while u >= 0:
            up += int(ev[u])
            u = int(parent[u])
        rows.append(up + int(cum[c + sub[c]] - cum[c]))
    return np.array(rows)


def run_shortlist(args):
    """Huge label sets: grouped labels scored through the shortlist
    (quail_classify_trie_tree_shortlist). One step = one call over all
    documents; metric = documents/s."""
    import numpy as np
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import bf16_tensor, kv_from_docs

    Q.build()
    sw = S.SHORTLIST_WORKLOADS[args.workload]
    w = S.with_docs(sw.base, args.docs) if args.docs else sw.base
    model = device_model(w.shape, 0)
    labels = S.make_labels(w, 0)
    K = len(labels.labels)
    G = sw.groups or (math.isqrt(K - 1) + 1)  # ceil(sqrt K)
    names = S.make_group_names(0, G, 1, w.shape.vocab)
    trie, _ = Q.Trie.grouped(labels.labels, labels.root_token, w.shape.vocab, names, num_groups=G)
    trie.upload()
    sl = Q.Shortlist(trie, 1)
    beam = sw.beam
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    N = w.num_docs
    ws = torch.empty(Q.workspace_size_shortlist(model, trie, sl, beam, N, docs.max_doc_len), dtype=torch.uint8,
                     device="cuda")
    lsc = torch.empty((N, K), device="cuda")
    prob = torch.empty((N, K), device="cuda")
    am = torch.empty((N,), dtype=torch.int32, device="cuda")
    sel = torch.empty((N, beam), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.classify_trie_tree_shortlist(model, kv, trie, sl, beam, N, ws, lsc, prob, am, sel, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    Q.device_status()
    launches_per_step = Q.launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    step()
    t1.record(stream)
    t1.synchronize()
    est_ms = t0.elapsed_time(t1)
    steps = args.steps if args.steps is not None else int(min(2000, max(20, 2000.0 / max(est_ms, 1e-3))))
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(steps)]
    for evs in stage_ev:
        for e in evs:
            e.record(stream)
    clocks = ClockSampler(str(torch.cuda.get_device_properties(0).pci_bus_id))
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hs = Q.STAGES.index("head")  # only the roofline kernel's events inside the timed loop
    start.record(stream)
    for k in range(steps):
        Q.set_stage_events([None] * (2 * hs) + stage_ev[k][2 * hs: 2 * hs + 2])
        step()
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    Q.set_stage_events(None)
    Q.device_status()
    elapsed_ms = start.elapsed_time(end)
    ms_per_step = elapsed_ms / steps
    value = N * steps / (elapsed_ms / 1e3)
    head_ms = statistics.mean(ev[2 * hs].elapsed_time(ev[2 * hs + 1]) for ev in stage_ev)
    bd_ev = stage_ev[:min(steps, 50)]  # stage breakdown, after the timed region
    torch.cuda.synchronize()
    for evs in bd_ev:
        Q.set_stage_events(evs)
        step()
    torch.cuda.synchronize()
    Q.set_stage_events(None)
    names5 = ("prefix_pass_select_layout", "prologue_attention", "wo_norm", "head", "scoring")
    stages_ms = {nm: statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for ev in bd_ev)
                 for i, nm in enumerate(names5)}

    # rows of the second pass: real (the kept groups' rows) and padded
    view = trie.view()
    grows = _group_rows(view, 1)
    selected = sel.cpu().numpy()
    real_rows = int(grows[selected].sum())
    pad_rows = N * beam * int(grows.max())

    # the flat trie_tree over the same grouped trie, for context (one timed call)
    flat_ms = None
    try:
        a = trie.n_eval
        wsf = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_TREE),
                          dtype=torch.uint8, device="cuda")
        Q.classify_trie_tree(model, kv, trie, N, wsf, lsc, prob, am, stream)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        Q.classify_trie_tree(model, kv, trie, N, wsf, lsc, prob, am, stream)
        f1.record(stream)
        f1.synchronize()
        flat_ms = f0.elapsed_time(f1)
        del wsf
        step()  # leave the shortlisted outputs in place
        torch.cuda.synchronize()
    except Q.QuailError:
        a = None

    # e2e: document KV from pinned host memory, every label's scores back
    e2e = None
    if not args.no_e2e:
        hk = bf16_tensor(docs.k_pool, "cpu").pin_memory()
        hv = bf16_tensor(docs.v_pool, "cpu").pin_memory()
        hpt = torch.from_numpy(docs.page_table).pin_memory()
        hdl = torch.from_numpy(docs.doc_len).pin_memory()
        o_ls = torch.empty((N, K)).pin_memory()
        o_pr = torch.empty((N, K)).pin_memory()
        o_am = torch.empty((N,), dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hk, hv, hpt, hdl))
        d2h = sum(t.numel() * t.element_size() for t in (o_ls, o_pr, o_am))

        kvs = [kv, kv_from_docs(docs)]  # two device KV buffers: copy one while the other computes

        def e2e_call(b):
            Q.classify_trie_tree_shortlist(model, kvs[b], trie, sl, beam, N, ws, lsc, prob, am, sel, stream)

        k_e2e = max(3, min(steps, int(3000.0 / max(est_ms + 3.0, 1e-3))))
        e2e_ms = timed_e2e(stream, [hk, hv, hpt, hdl], [list(x.tensors) for x in kvs], e2e_call,
                           [(lsc, o_ls), (prob, o_pr), (am, o_am)], k_e2e)
        e2e = e2e_entry(N, k_e2e, e2e_ms, h2d, d2h, [hk, hv, hpt, hdl], list(kvs[1].tensors))

    # roofline: the second pass's output-head GEMM, FLOPs of the real rows
    peaks = measured_peaks()
    d, V = w.shape.hidden, w.shape.vocab
    flops = 2.0 * d * V * real_rows
    achieved = flops / (head_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "traffic": recorded_traffic(sw.name, real_rows, "lm_head_gemm_shortlist_traffic.json"),
                "kernel": "umma_gemm_kernel<EpiHead> (second pass)", "head_ms": head_ms,
                "real_rows": real_rows, "padded_rows": pad_rows,
                "peak_kind": f"bf16 burst ({peaks['source']})",
                "note": "FLOPs of the kept groups' rows; padding rows (copies of the root) are extra work"}
    kv_bytes = float(docs.doc_len.sum()) * w.shape.n_kv_heads * w.shape.head_dim * 2 * 2
    path_bytes = 2 * kv_bytes + 2 * 2.0 * d * V
    path_flops = 2.0 * d * V * (N + real_rows)
    t_b = path_bytes / (peaks["hbm_gbs"] * 1e9)
    t_f = path_flops / (peaks["bf16_tflops"] * 1e12)
    path = {"t_bytes_us": t_b * 1e6, "t_flops_us": t_f * 1e6, "t_star_us": max(t_b, t_f) * 1e6,
            "ms_per_step": ms_per_step, "frac": max(t_b, t_f) * 1e3 / ms_per_step}

    cpu = None
    if not args.no_cpu_baseline:
        from oracle import shortlist as OSL
        from oracle.trie import build_trie
        rw = OSL.rewrite_grouped(labels.labels, names, OSL.group_labels(labels.labels, G))
        ref_t = build_trie(rw, labels.root_token, V)
        L = oracle_layer(w.shape, 0)
        L.lm_head()
        c0 = time.perf_counter()
        done = 0
        while done < N and (done == 0 or time.perf_counter() - c0 < 15.0):
            dk_, dv_ = oracle_doc_kv(docs, done)
            OSL.shortlist(L, dk_, dv_, ref_t, 1, beam)
            done += 1
        sec = time.perf_counter() - c0
        cpu = {"value": done / sec, "unit": "docs/s", "cores": cores(), "kind": "oracle",
               "sample": f"first {done} documents of {w.name} ({sec:.1f} s, oracle shortlist with the same "
                         f"groups and beam)"}
    out = {
        "metric": "documents classified/sec at 1 GB300 (shortlisted trie_tree over grouped labels)",
        "value": value, "unit": "docs/s", "n_gpus": 1, "steps": steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": sw.name, "docs_per_gpu": N, "labels": K, "groups": G, "beam": beam,
                   "trie_nodes": trie.n_nodes, "eval_positions_flat": a, "second_pass_rows": real_rows,
                   "second_pass_rows_padded": pad_rows, "hidden": d, "vocab": V,
                   "l2": "inputs larger than L2 (output head 0.78 GB read twice per step)",
                   "parallelism": "one replica (documents shard across GPUs with no collective)"},
        "roofline": roofline, "path_roofline": path, "stages_ms": stages_ms,
        "flat_trie_tree_ms": flat_ms, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * steps, "clocks": clk,
    }
    print(json.dumps(out), flush=True)


def _timed_loop(stream, steps, call, n_stage_events=0, keep=None):
    """K calls between CUDA events on `stream`, synchronize on both
    sides; per-call stage events when n_stage_events > 0, of which only the
    indices in `keep` are handed to the library when given (an event between
    two kernels keeps the second from launching early). Returns
    (elapsed ms, stage events per call, clocks)."""
    import torch

    import trie_label_scoring_gb300 as Q
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_stage_events)] for _ in range(steps)]
    for evs in stage_ev:
        for e in evs:
            e.record(stream)
    clocks = ClockSampler(str(torch.cuda.get_device_properties(torch.cuda.current_device()).pci_bus_id))
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        if n_stage_events:
            evs = stage_ev[k]
            Q.set_stage_events(evs if keep is None else [e if i in keep else None for i, e in enumerate(evs)])
        call()
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    Q.set_stage_events(None)
    Q.device_status()
    return start.elapsed_time(end), stage_ev, clk


def run_letters(args):
    """The letters variant ("To Classify, Try a Trie Tree", sec. 3.3): one
    answer position per document scored against the letter tokens
    (quail_classify_letters). One step = one call over all documents."""
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs

    Q.build()
    w = S.WORKLOADS[args.workload]
    if args.docs:
        w = S.with_docs(w, args.docs)
    model = device_model(w.shape, 0)
    letters = S.make_labels(w, 0)
    tokens = [l[0] for l in letters.labels]
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    N, M = w.num_docs, len(tokens)
    ws = torch.empty(Q.workspace_size(model, None, M, N, docs.max_doc_len, Q.MODE_LETTERS), dtype=torch.uint8,
                     device="cuda")
    lp = torch.empty((N, M), device="cuda")
    pr = torch.empty((N, M), device="cuda")
    am = torch.empty((N,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        Q.classify_letters(model, kv, tokens, letters.root_token, N, ws, lp, pr, am, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    Q.device_status()
    launches = Q.launch_count()
    steps = args.steps if args.steps is not None else 200
    ai = Q.STAGES.index("attention")
    elapsed_ms, stage_ev, clk = _timed_loop(stream, steps, step, 10, keep=(2 * ai, 2 * ai + 1))
    attention_ms = statistics.mean(ev[2 * ai].elapsed_time(ev[2 * ai + 1]) for ev in stage_ev)
    bd_ev = stage_ev[:min(steps, 20)]  # stage breakdown, after the timed region
    for evs in bd_ev:
        Q.set_stage_events(evs)
        step()
    torch.cuda.synchronize()
    Q.set_stage_events(None)
    stages_ms = {name: statistics.mean(ev[2 * i].elapsed_time(ev[2 * i + 1]) for ev in bd_ev)
                 for i, name in enumerate(Q.STAGES[:4])}
    ms = elapsed_ms / steps
    peaks = measured_peaks()
    kv_bytes = float(docs.doc_len.sum()) * w.shape.n_kv_heads * w.shape.head_dim * 2 * 2
    att = kv_bytes / (attention_ms / 1e3) / 1e9
    t_kv = kv_bytes / (peaks["hbm_gbs"] * 1e9)
    out = {
        "metric": "documents classified/sec at 1 GB300 (letters)", "value": N * steps / (elapsed_ms / 1e3),
        "unit": "docs/s", "n_gpus": 1, "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": w.name, "docs_per_gpu": N, "letters": M, "doc_tokens_per_gpu": int(docs.doc_len.sum()),
                   "l2": "doc KV %.2f GB per step" % (kv_bytes / 1e9),
                   "parallelism": "one replica (documents shard across GPUs with no collective)"},
        "roofline": {"bound": "hbm", "achieved": att, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": att / peaks["hbm_gbs"], "traffic": None, "kernel": "doc attention (one row per document)",
                     "attention_ms": attention_ms, "peak_kind": f"HBM copy ({peaks['source']})"},
        "path_roofline": {"t_kv_us": t_kv * 1e6, "ms_per_step": ms, "frac": t_kv * 1e3 / ms},
        "stages_ms": stages_ms, "cpu_baseline": None, "e2e": None, "gpu_launches": launches * steps,
        "clocks": clk,
    }
    print(json.dumps(out), flush=True)


def run_decode(args):
    """Greedy trie_decode ("To Classify, Try a Trie Tree", sec. 3.1) over a
    tree workload: one step of the bench = the decode steps it takes for every
    document to reach a label (quail_classify_trie_decode_step, called that
    many times; the count is fixed in the warm-up, so no host read happens
    inside the timed region)."""
    import torch

    import synthetic as S
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs

    Q.build()
    w = S.WORKLOADS[args.workload]
    if args.docs:
        w = S.with_docs(w, args.docs)
    model = device_model(w.shape, 0)
    labels = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    trie = Q.Trie(labels.labels, labels.root_token, w.shape.vocab, labels.continuation)
    trie.upload()
    N = w.num_docs
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_DECODE), dtype=torch.uint8,
                     device="cuda")
    cur = torch.zeros(N, dtype=torch.int32, device="cuda")
    lab = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    act = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    n_steps = 0
    while True:  # warm-up: how many decode steps this batch takes
        Q.classify_trie_decode_step(model, kv, trie, N, cur, lab, act, ws, None, stream)
        n_steps += 1
        if int(act.item()) == 0 or n_steps >= 64:
            break
    launches_per_step_call = Q.launch_count()

    def decode():
        cur.zero_()
        lab.fill_(-1)
        for _ in range(n_steps):
            Q.classify_trie_decode_step(model, kv, trie, N, cur, lab, act, ws, None, stream)

    for _ in range(max(args.warmup, 3)):
        decode()
    Q.device_status()
    steps = args.steps if args.steps is not None else 100
    elapsed_ms, _, clk = _timed_loop(stream, steps, decode)
    ms = elapsed_ms / steps
    peaks = measured_peaks()
    kv_bytes = float(docs.doc_len.sum()) * w.shape.n_kv_heads * w.shape.head_dim * 2 * 2
    out = {
        "metric": "documents classified/sec at 1 GB300 (greedy trie_decode)",
        "value": N * steps / (elapsed_ms / 1e3), "unit": "docs/s", "n_gpus": 1, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, random-init weights)",
        "config": {"workload": w.name, "docs_per_gpu": N, "labels": len(labels.labels),
                   "decode_steps": n_steps, "doc_tokens_per_gpu": int(docs.doc_len.sum()),
                   "parallelism": "one replica (documents shard across GPUs with no collective)"},
        "roofline": {"bound": "hbm", "achieved": n_steps * kv_bytes / (ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": n_steps * kv_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": None, "kernel": "whole decode (document KV re-read at every step)",
                     "peak_kind": f"HBM copy ({peaks['source']})",
                     "note": "the bytes are those of all documents at every step; decided documents skip "
                             "their attention, so this overstates the work of the later steps"},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": launches_per_step_call * n_steps * steps, "clocks": clk,
    }
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.oracle_rate:
        run_oracle_rate(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    gpu_setup(args)
    import synthetic as S
    if args.workload in S.ML_WORKLOADS:  # the whole decoder stack
        run_ml(args)
    elif args.workload in S.SHORTLIST_WORKLOADS:  # grouped labels through the shortlist
        run_shortlist(args)
    elif "-join" in args.workload:  # AI.IF join workloads (synthetic labels kind "join")
        run_join(args)
    elif "-letters" in args.workload:  # the letters variant
        run_letters(args)
    elif args.decode:  # greedy trie_decode on a tree workload
        run_decode(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
