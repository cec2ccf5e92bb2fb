"""Benchmark of the KPool indexer selection on synthetic GLM-shaped inputs.

One step = one kpool_select call (plan, pool, score+select, expand) over the
whole batch. Default workload: the pages-scale causal batch, 1 x 524288 tokens,
32 index heads, d = 128, kpool 4, index_topk 2048 (budget 512 pools), bf16 q/k,
fp32 head weights -- the configuration the pages quote their selection time on.

Prints one JSON line (rank 0). `value` is whole-job throughput in scored
(query row, eligible pool) pairs per second with inputs resident in HBM;
`e2e` is the same metric through the C ABI with host (pinned) buffers and the
host<->device copies inside the timed region. `roofline` reports the
score+select kernel against the measured bf16 tensor-core peak, timed with CUDA
events that the library records around each of its kernels. `cpu_baseline` is
the CPU oracle timed on a bounded row sample on this host's cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU: replicas only -- every rank runs its own copy of the workload (the
selection has no exchange step on one node), barrier + max-over-ranks timing,
value = all ranks' pairs / max time.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_kpool_gb300 import build as kbuild  # noqa: E402
from sparse_attention_kpool_gb300 import kpool as K  # noqa: E402
from sparse_attention_kpool_gb300 import workloads as W  # noqa: E402

METRIC = "KPool selection sec @512k tokens; scored pairs/s; % of bf16 tensor-core peak"
UNIT = "scored pairs/s"
FLOP_PER_PAIR_PER_HEAD_DIM = 2  # one multiply-add per (head, channel) of a scored pair
# The pages' unsharded KPool selection microbenchmark at 512k tokens per sequence,
# seconds per rank (NVIDIA/Megatron-LM pull request #8299, "Validation (from SkyRL)").
PAGES_SEC_512K = 21.07

# DRAM traffic of the score+select kernel from one ncu capture, per launch at the
# pages-scale workload, tied to the kernel source it was measured on: when the
# source hash differs the number is stale and is reported as null.
NCU_TRAFFIC = {"kernel_sha256": "8c12fac7b912701f", "workload": "pages_512k",
               # long_128k capture: 1.100543 GB read + 0.212087 GB written per launch; q, w and the
               # pool ids grow with the rows, so x4 at 524288 tokens
               "bytes_per_launch": 4 * (1100542976 + 212086784)}
# The same for the index-score mode of that kernel, per launch of the long_128k chunked run
# (the mean over one step's 8 chunk launches: 1.130 GB read, 16.668 GB written in all).
NCU_TRAFFIC_SCORES = {"kernel_sha256": "8c12fac7b912701f", "workload": "long_128k",
                      "bytes_per_launch": (1129766656 + 16667923712) / 8}
# And for the decode rows' score kernel (kpool_rows.cu), per launch at decode_262k (the mean
# over three launches).
NCU_TRAFFIC_ROWS = {"kernel_sha256": "874a5f90baaa7d8a", "workload": "decode_262k",
                    "bytes_per_launch": (806049024 + 8812800) / 3}


def source_sha(path: str) -> str:
    """Hash of a CUDA source's code with comments and blank lines removed, so a comment
    edit does not invalidate counters taken on the same code."""
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "_source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.device_index = device_index

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        bus = _pci_bus_id(self.device_index)
        if bus:
            cmd += ["-i", bus]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _pci_bus_id(dev: int):
    try:
        p = torch.cuda.get_device_properties(dev)
        dom, bus, d = getattr(p, "pci_domain_id", None), getattr(p, "pci_bus_id", None), getattr(p, "pci_device_id", None)
        if bus is None:
            return None
        return f"{dom or 0:08X}:{bus:02X}:{d or 0:02X}.0"
    except Exception:
        return None


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(dev_inputs: dict, wl: W.Workload, rows: np.ndarray, kp=None):
    """Time the CPU oracle on the listed rows (the bounded CPU baseline sample)."""
    from oracle import oracle
    from tests import parity
    cu = dev_inputs["cu_seqlens"].cpu().numpy()
    k_bits = parity.bits(dev_inputs["k"])
    ridx = torch.as_tensor(rows, device=dev_inputs["q"].device)
    q_rows = parity.bits(dev_inputs["q"][ridx])
    w_rows = dev_inputs["w"][ridx].cpu().numpy()
    t0 = time.perf_counter()
    if kp is None:
        kp = oracle.pool(k_bits, wl.dtype, cu, wl.kpool)
    out = oracle.select(q_rows, w_rows, kp, cu, rows, wl.dtype, wl.kpool, wl.index_topk, wl.scale)
    dt = time.perf_counter() - t0
    pairs = int(out["eligible"].sum())
    return {"seconds": dt, "pairs": pairs, "threads": oracle.threads(), "out": out, "kp": kp}


def pick_sample_rows(wl: W.Workload, target_pairs: float, seed: int) -> np.ndarray:
    """Uniform rows until their eligible-pool count reaches target_pairs."""
    rng = np.random.default_rng(seed)
    T = wl.total_tokens
    cu = wl.cu_seqlens().numpy()
    rows, pairs = [], 0
    while pairs < target_pairs and len(rows) < T:
        r = int(rng.integers(0, T))
        b = int(np.searchsorted(cu, r, side="right") - 1)
        pairs += (r - int(cu[b]) + 1) // wl.kpool
        rows.append(r)
    return np.array(sorted(set(rows)), dtype=np.int64)


def workload_config(wl: W.Workload, world: int) -> dict:
    """The `config` object of the JSON line, identical for both arms."""
    return {"workload": wl.name, "seqlens": list(wl.seqlens) if len(wl.seqlens) <= 8 else wl.num_seqs,
            "heads": wl.heads, "head_dim": wl.head_dim, "kpool": wl.kpool, "index_topk": wl.index_topk,
            "budget": wl.budget, "scale": wl.scale,
            "inputs": "q,k %s N(0,1), w fp32 U(0,1), seeded (CUDA Philox)" % wl.dtype,
            "l2": "inputs larger than L2 (q alone is %.1f GiB)" % (wl.total_tokens * wl.heads * wl.head_dim * 2 / 2**30),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def reference_arm(args, wl, world, rank):
    """The oracle as the reference implementation: each step scores a bounded row sample."""
    if rank != 0:
        return
    torch.manual_seed(0)
    inp = W.generate(wl, "cpu" if not torch.cuda.is_available() else "cuda")
    from oracle import oracle
    oracle.build()
    cu = inp["cu_seqlens"].cpu().numpy()
    from tests import parity
    kp = oracle.pool(parity.bits(inp["k"]), wl.dtype, cu, wl.kpool)
    times, pairs_all = [], []
    for step in range(args.warmup + args.steps):
        rows = pick_sample_rows(wl, args.ref_pairs_per_step, seed=1000 + step)
        res = oracle_sample(inp, wl, rows, kp=kp)
        if step >= args.warmup:
            times.append(res["seconds"])
            pairs_all.append(res["pairs"])
    total_t, total_p = sum(times), sum(pairs_all)
    value = total_p / total_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, world),
        "sec_per_selection_extrapolated": wl.causal_pairs() / value,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{len(times)} steps x ~{args.ref_pairs_per_step:.2e} pairs of uniform rows "
                                   f"of {wl.name}; seconds/selection extrapolated by pair count"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def rows_traffic(wl) -> float | None:
    """DRAM bytes per launch of the decode score kernel from the ncu capture, while the
    kernel source is the one that was captured and the workload the captured one."""
    src = os.path.join(ROOT, "sparse_attention_kpool_gb300", "csrc", "kpool_rows.cu")
    t = NCU_TRAFFIC_ROWS
    return t["bytes_per_launch"] if t["kernel_sha256"] == source_sha(src) and t["workload"] == wl.name else None


def rows_config(wl: W.RowsWorkload, world: int) -> dict:
    return {"workload": wl.name, "key_seqlens": list(wl.seqlens) if len(set(wl.seqlens)) > 1 else
            f"{len(wl.seqlens)} x {wl.seqlens[0]}", "rows": wl.num_rows, "heads": wl.heads,
            "head_dim": wl.head_dim, "kpool": wl.kpool, "index_topk": wl.index_topk, "budget": wl.budget,
            "scale": wl.scale, "inputs": "k, q bf16 N(0,1), w fp32 U(0,1), seeded (CUDA Philox)",
            "l2": "pooled keys of all rows' sequences (%.0f MiB) exceed L2; a 256 MiB read flushes it "
                  "between steps" % (wl.total_tokens // wl.kpool * wl.head_dim * 2 / 2**20),
            "parallelism": "replicas" if world > 1 else "single GPU"}


ROWS_METRIC = "KPool decode selection: scored pairs/s (rows against a pooled-key cache)"


def rows_bench(args, wl: W.RowsWorkload, world: int, rank: int, emit: bool = True):
    """Decode / short-query path: kpool_select_rows against a resident pooled-key cache.
    Prints the JSON line on rank 0 when `emit`, and returns it."""
    if args.impl == "reference":
        if rank == 0:
            from oracle import oracle
            from tests import parity
            oracle.build()
            inp = W.generate_rows(wl, "cuda" if torch.cuda.is_available() else "cpu")
            cu = inp["cu_seqlens"].cpu().numpy()
            kp = oracle.pool(parity.bits(inp["k"]), wl.dtype, cu, wl.kpool)
            qb, wb = parity.bits(inp["q"]), inp["w"].cpu().numpy()
            rows = np.array(wl.global_rows(), dtype=np.int64)
            times = []
            for i in range(args.warmup + args.steps):
                t0 = time.perf_counter()
                oracle.select(qb, wb, kp, cu, rows, wl.dtype, wl.kpool, wl.index_topk, wl.scale)
                if i >= args.warmup:
                    times.append(time.perf_counter() - t0)
            v = wl.scored_pairs() / statistics.median(times)
            print(json.dumps({"impl": "reference", "metric": ROWS_METRIC, "value": v, "unit": UNIT, "n_gpus": world,
                              "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                              "config": rows_config(wl, world),
                              "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                                               "sample": f"all {wl.num_rows} rows, pooling excluded"},
                              "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                  flush=True)
        return
    kbuild.build()
    K.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    inp = W.generate_rows(wl, dev)
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)  # the cache exists before decoding
    R, B, Wd = wl.num_rows, wl.budget, wl.width
    ids = torch.empty((R, B), dtype=torch.int32, device=dev)
    toks = torch.empty((R, Wd), dtype=torch.int32, device=dev)
    ws = K.new_rows_workspace(R, wl.total_tokens, wl.num_seqs, wl.kpool, wl.index_topk, dev)
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for evs in step_events:
        for e in evs:
            e.record(stream)

    def step(ev=None, q=inp["q"], w=inp["w"], rs=inp["row_seq"], rp=inp["row_pos"]):
        K.kpool_select_rows(q, w, rs, rp, kp, inp["cu_seqlens"], wl.total_tokens, wl.kpool, wl.index_topk,
                            wl.scale, out_pool_ids=ids, out_token_ids=toks, workspace=ws, stream=stream,
                            stage_events=ev)

    for _ in range(args.warmup):
        step(step_events[0])
    torch.cuda.synchronize()
    if K.kpool_last_device_error(ws) != K.KPOOL_OK:
        raise K.KpoolError(K.kpool_last_device_error(ws), "device")
    # a read of 256 MiB (twice L2) between steps, so every step reads the key cache from
    # HBM; a read leaves no dirty lines whose write-back would land in the next step
    flush = torch.ones(64 << 20, dtype=torch.int32, device=dev)

    def flush_l2():
        return flush.max()
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    per_step = []
    for s_i in range(args.steps):
        flush_l2()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(step_events[s_i])
        b.record(stream)
        per_step.append((a, b))
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    ms = statistics.median([a.elapsed_time(b) for a, b in per_step])
    # the same step captured once in a CUDA graph and replayed (what a decode loop would do)
    graph_ms = None
    k_ms_graph = None
    try:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        g_ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in g_ev:
            e.record(stream)
        # `graph` is the step a decode loop replays; `graph_ev` the same step with the stage
        # events as event-record nodes (they lengthen the graph), for the per-kernel times
        graph, graph_ev = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            for g, evs in ((graph, None), (graph_ev, g_ev)):
                with torch.cuda.graph(g, stream=gs):
                    K.kpool_select_rows(inp["q"], inp["w"], inp["row_seq"], inp["row_pos"], kp, inp["cu_seqlens"],
                                        wl.total_tokens, wl.kpool, wl.index_topk, wl.scale, out_pool_ids=ids,
                                        out_token_ids=toks, workspace=ws, stream=gs, stage_events=evs)
        stream.wait_stream(gs)
        g_t = []
        for s_i in range(args.warmup + args.steps):
            flush_l2()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            g_t.append((a, b))
        torch.cuda.synchronize()
        graph_ms = statistics.median([a.elapsed_time(b) for a, b in g_t[args.warmup:]])
        # per-kernel times from the graph's own event nodes (no host launch gaps): one
        # replay at a time, its stage events read before the next replay records them again
        g_k = []
        for s_i in range(args.steps):
            flush_l2()
            graph_ev.replay()
            torch.cuda.synchronize()
            g_k.append([g_ev[i].elapsed_time(g_ev[i + 1]) for i in range(3)])
        k_ms_graph = [statistics.median([x[i] for x in g_k]) for i in range(3)]
    except RuntimeError as ex:  # graph capture unavailable: report the eager number only
        print(f"graph capture skipped: {ex}", file=sys.stderr)
    ms_step = max_over_ranks(ms, world)
    k_ms_eager = [statistics.median([evs[i].elapsed_time(evs[i + 1]) for evs in step_events]) for i in range(3)]
    k_ms = k_ms_graph if k_ms_graph is not None else k_ms_eager
    pairs = wl.scored_pairs()
    value = world * pairs / (ms_step / 1e3)
    # e2e: the rows' inputs come from pinned host memory, the selection goes back to it
    h = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in ("q", "w", "row_seq", "row_pos")}
    for k2 in h:
        h[k2].copy_(inp[k2])
    d = {k2: torch.empty_like(inp[k2]) for k2 in h}
    h_ids = torch.empty(ids.shape, dtype=ids.dtype, pin_memory=True)
    h_toks = torch.empty(toks.shape, dtype=toks.dtype, pin_memory=True)
    bi = sum(v.numel() * v.element_size() for v in h.values())
    bo = h_ids.numel() * 4 + h_toks.numel() * 4
    e2e_t = []
    for _ in range(args.warmup + args.steps):
        flush_l2()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k2 in d:
            d[k2].copy_(h[k2], non_blocking=True)
        step(None, d["q"], d["w"], d["row_seq"], d["row_pos"])
        h_ids.copy_(ids, non_blocking=True)
        h_toks.copy_(toks, non_blocking=True)
        b.record(stream)
        e2e_t.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(statistics.median([a.elapsed_time(b) for a, b in e2e_t[args.warmup:]]), world)
    peaks = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    H, dd = wl.heads, wl.head_dim
    score_bytes = pairs * dd * 2 + R * H * dd * 2 + R * H * 4 + pairs * 4  # pooled keys, q, w in; scores out
    achieved = score_bytes / (k_ms[1] / 1e3) / 1e9
    line = {
        "metric": ROWS_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": rows_config(wl, world),
        "us_per_decode_step": 1e3 * ms_step,
        "us_per_decode_step_graph": None if graph_ms is None else 1e3 * graph_ms,
        "kernel_ms": {"plan": k_ms[0], "score": k_ms[1], "select": k_ms[2],
                      "timed": "graph replay" if k_ms_graph is not None else "eager"},
        "kernel_ms_eager": {"plan": k_ms_eager[0], "score": k_ms_eager[1], "select": k_ms_eager[2]},
        "roofline": {"kernel": "rows_score_kernel", "bound": "hbm", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": rows_traffic(wl),
                     "peak_kind": f"HBM copy, {peaks['_source']}", "algorithmic_bytes_per_launch": score_bytes},
        "clocks": clock_info, "gpu_launches": 4 * args.steps,
        "e2e": {"value": world * pairs / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms},
    }
    if rank == 0 and not args.no_cpu:
        from oracle import oracle
        from tests import parity
        cu = inp["cu_seqlens"].cpu().numpy()
        kpo = oracle.pool(parity.bits(inp["k"]), wl.dtype, cu, wl.kpool)
        rows = np.array(wl.global_rows(), dtype=np.int64)
        t0 = time.perf_counter()
        ref = oracle.select(parity.bits(inp["q"]), inp["w"].cpu().numpy(), kpo, cu, rows, wl.dtype, wl.kpool,
                            wl.index_topk, wl.scale)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": pairs / dt, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                                "sample": f"all {R} rows ({pairs:.3e} pairs, {dt:.2f} s, pooling excluded)"}
        ok = True
        try:
            ref["kp"], ref["rows"] = kpo, rows
            parity.compare_float({"cu_seqlens": inp["cu_seqlens"]}, wl, ref, ids.cpu().numpy(), None,
                                 toks.cpu().numpy(), q_rows=inp["q"], w_rows=inp["w"])
        except AssertionError as ex:
            ok = False
            line["parity_sample_error"] = str(ex)[:200]
        line["parity_sample"] = {"rows": R, "ok": ok}
    if rank == 0 and emit:
        print(json.dumps(line), flush=True)
    return line


SCORES_METRIC = "KPool index scores: scored pairs/s (full masked [rows, pools] fp32 scores, row chunks <= 2 GiB)"
# The pages compute their index scores in row chunks of at most 2 GiB (NVIDIA/Megatron-LM
# pull request #8299, "Change"); the benchmark chunks the same way.
SCORE_CHUNK_BYTES = 2 << 30


def scores_config(wl: W.Workload, world: int, ld: int, chunk: int, nck: int) -> dict:
    c = workload_config(wl, world)
    c.update({"ld": ld, "chunk_rows": chunk, "chunks": nck,
              "output": "fp32 [rows, ld] per chunk into one reused device buffer",
              "l2": "inputs larger than L2 (q %.1f GiB, each chunk's output %.1f GiB)" % (
                  wl.total_tokens * wl.heads * wl.head_dim * 2 / 2**30, chunk * ld * 4 / 2**30)})
    c.pop("index_topk")
    c.pop("budget")
    return c


def index_scores_bench(args, wl: W.Workload, world: int, rank: int, emit: bool = True):
    """Full index scores of every row (kpool_pool_keys once, then kpool_index_scores_pooled
    per row chunk of <= 2 GiB of output). Prints the JSON line on rank 0 when `emit`, and
    returns it."""
    kbuild.build()
    K.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    inp = W.generate(wl, dev)
    T, H, d = wl.total_tokens, wl.heads, wl.head_dim
    ld = max(1, max(int(L) // wl.kpool for L in wl.seqlens))  # the widest row any sequence has
    chunk = max(1, min(T, SCORE_CHUNK_BYTES // (4 * ld)))
    bounds = list(range(0, T, chunk)) + [T]
    nck = len(bounds) - 1
    dt_code = K.KPOOL_BF16 if wl.dtype == "bf16" else K.KPOOL_F32
    ws = K.new_workspace(T, wl.num_seqs, H, d, dt_code, wl.kpool, 0, dev)
    out = [torch.empty((chunk, ld), dtype=torch.float32, device=dev)]
    if not args.no_e2e:
        out.append(torch.empty((chunk, ld), dtype=torch.float32, device=dev))  # double buffer for the downloads
    kp = torch.empty((max(1, T // wl.kpool), d), dtype=inp["k"].dtype, device=dev)
    pairs = wl.causal_pairs()
    flops = FLOP_PER_PAIR_PER_HEAD_DIM * H * d * pairs
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(nck)]
          for _ in range(args.steps)]
    for s_ev in ev:
        for c_ev in s_ev:
            for e in c_ev:
                e.record(stream)

    def step(evs=None, x=inp, on_chunk=None):
        K.kpool_pool_keys(x["k"], x["cu_seqlens"], wl.kpool, out=kp, workspace=ws, stream=stream)
        for c in range(nck):
            lo, hi = bounds[c], bounds[c + 1]
            buf = out[c % 2] if on_chunk is not None else out[0]
            K.kpool_index_scores(x["q"], kp, x["w"], x["cu_seqlens"], wl.kpool, wl.scale, ld=ld, out=buf[:hi - lo],
                                 row_range=(lo, hi), workspace=ws, stream=stream, pooled=True,
                                 stage_events=None if evs is None else evs[c])
            if on_chunk is not None:
                on_chunk(c, buf[:hi - lo])

    for _ in range(args.warmup):
        step(ev[0])
    torch.cuda.synchronize()
    st = K.kpool_last_device_error(ws)
    if st != K.KPOOL_OK:
        raise K.KpoolError(st, "device (index scores)")
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    per = []
    for s_i in range(args.steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(ev[s_i])
        b.record(stream)
        per.append((a, b))
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop()
    ms_step = max_over_ranks(statistics.median([a.elapsed_time(b) for a, b in per]), world)
    value = world * pairs / (ms_step / 1e3)
    k_ms = statistics.median([sum(c[2].elapsed_time(c[3]) for c in s_ev) for s_ev in ev])  # score kernels
    setup_ms = statistics.median([sum(c[0].elapsed_time(c[2]) for c in s_ev) for s_ev in ev])  # plans
    peaks = measured_peaks()
    peak_burst = float(peaks["bf16_tflops"])
    peak_sust = float(peaks.get("bf16_tflops_sustained", peak_burst))
    hbm = float(peaks["hbm_gbs"])
    achieved = flops / (k_ms / 1e3) / 1e12
    out_bytes = T * ld * 4
    alg_bytes = T * H * d * 2 + T * H * 4 + wl.num_pools() * d * 2 + out_bytes  # q, w, pooled keys in; scores out

    # end to end: inputs from pinned host memory, every chunk's scores back to one pinned host
    # buffer; chunk c+1 computes while chunk c downloads on a copy stream (two device buffers)
    e2e = None
    if not args.no_e2e:
        keys = ("q", "k", "w", "cu_seqlens")
        h_in = {k2: torch.empty(inp[k2].shape, dtype=inp[k2].dtype, pin_memory=True) for k2 in keys}
        for k2 in keys:
            h_in[k2].copy_(inp[k2])
        d_in = {k2: torch.empty_like(inp[k2]) for k2 in keys}
        h_out = torch.empty((chunk, ld), dtype=torch.float32, pin_memory=True)
        copy = torch.cuda.Stream(device=dev)
        bi = sum(v.numel() * v.element_size() for v in h_in.values())
        freed = [None, None]  # event: the download of buffer i finished

        def download(c, buf):
            done = torch.cuda.Event()
            done.record(stream)
            copy.wait_event(done)
            with torch.cuda.stream(copy):
                h_out[:buf.shape[0]].copy_(buf, non_blocking=True)
                f = torch.cuda.Event()
                f.record(copy)
            freed[c % 2] = f
            nxt = freed[(c + 1) % 2]
            if nxt is not None:
                stream.wait_event(nxt)  # chunk c+1 writes the buffer chunk c-1 was downloaded from

        e2e_t = []
        for i in range(args.warmup + args.steps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k2 in keys:
                d_in[k2].copy_(h_in[k2], non_blocking=True)
            freed[0] = freed[1] = None
            step(None, d_in, download)
            stream.wait_stream(copy)
            b.record(stream)
            e2e_t.append((a, b))
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(statistics.median([a.elapsed_time(b) for a, b in e2e_t[args.warmup:]]), world)
        e2e = {"value": world * pairs / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": out_bytes, "ms_per_step": e2e_ms,
               "d2h_GB/s": out_bytes / (e2e_ms / 1e3) / 1e9,
               "pipelining": "each chunk's scores download on a copy stream while the next chunk computes"}
        del h_in, d_in, h_out
    line = {
        "metric": SCORES_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": scores_config(wl, world, ld, chunk, nck),
        "kernel_ms": {"plans": setup_ms, "index_scores": k_ms, "launches_per_step": nck},
        "roofline": {"kernel": "select_tc_kernel (index-score mode)", "bound": "tensor", "achieved": achieved,
                     "peak": peak_burst, "unit": "TFLOP/s", "frac": achieved / peak_burst, "traffic": None,
                     "peak_kind": f"bf16 burst, {peaks['_source']}", "frac_of_sustained": achieved / peak_sust,
                     "algorithmic_flop_per_launch": flops / nck, "algorithmic_bytes_per_launch": alg_bytes / nck,
                     "output_GB/s": out_bytes / (k_ms / 1e3) / 1e9,
                     "output_frac_of_hbm": out_bytes / (k_ms / 1e3) / 1e9 / hbm,
                     "note": "per launch = the step's total over its chunk launches / launches"},
        "clocks": clock_info,
        "gpu_launches": (2 + 2 * nck) * args.steps,
        "e2e": e2e,
    }
    traffic = NCU_TRAFFIC_SCORES
    tc_src = os.path.join(ROOT, "sparse_attention_kpool_gb300", "csrc", "kpool_select_tc.cu")
    if traffic["kernel_sha256"] == source_sha(tc_src) and traffic["workload"] == wl.name:
        line["roofline"]["traffic"] = traffic["bytes_per_launch"]
    if rank == 0 and not args.no_cpu:
        from oracle import oracle
        from tests import parity
        oracle.build()
        rows = pick_sample_rows(wl, args.cpu_sample_pairs / 4, seed=11)
        cu = inp["cu_seqlens"].cpu().numpy()
        kpo = oracle.pool(parity.bits(inp["k"]), wl.dtype, cu, wl.kpool)
        t0 = time.perf_counter()
        ref = parity.oracle_full_scores(inp, wl, rows, ld, kp=kpo)
        dt = time.perf_counter() - t0
        sp = int(np.isfinite(ref).sum())
        line["cpu_baseline"] = {"value": sp / dt, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                                "sample": f"{len(rows)} uniform rows of {wl.name} ({sp:.3e} pairs, {dt:.1f} s, "
                                          f"pooling excluded); fp64 scores"}
        # the same rows as a parity spot check: each through its own one-row call
        one = torch.empty((1, ld), dtype=torch.float32, device=dev)
        got = np.empty((len(rows), ld), dtype=np.float32)
        K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool, out=kp, workspace=ws, stream=stream)
        for i, r in enumerate(rows):
            K.kpool_index_scores(inp["q"], kp, inp["w"], inp["cu_seqlens"], wl.kpool, wl.scale, ld=ld, out=one,
                                 row_range=(int(r), int(r) + 1), workspace=ws, stream=stream, pooled=True)
            got[i] = one.cpu().numpy()
        ok = True
        try:
            err = parity.compare_full_scores(got, ref, exact=wl.values == "integer", what=wl.name)
            line["parity_sample"] = {"rows": int(len(rows)), "ok": True, "max_rel_err": err}
        except AssertionError as ex:
            line["parity_sample"] = {"rows": int(len(rows)), "ok": False, "error": str(ex)[:200]}
    if rank == 0 and emit:
        print(json.dumps(line), flush=True)
    del out, kp, inp, ws
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="pages_512k", choices=sorted(W.BY_NAME) + sorted(W.ROWS_BY_NAME))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-pairs", type=float, default=4.0e7,
                    help="eligible pairs in the CPU oracle's timed row sample")
    ap.add_argument("--ref-pairs-per-step", type=float, default=1.5e7)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode workload that the default (pages-scale) run also measures")
    ap.add_argument("--index-scores", action="store_true",
                    help="measure the full index-score output (kpool_index_scores) on --workload instead")
    ap.add_argument("--no-index-scores", action="store_true",
                    help="skip the index-score measurement that the default (pages-scale) run also makes")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.workload in W.ROWS_BY_NAME:
        rows_bench(args, W.ROWS_BY_NAME[args.workload], world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    wl = W.BY_NAME[args.workload]
    if args.index_scores and args.impl == "ours":
        index_scores_bench(args, wl, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.impl == "reference":
        reference_arm(args, wl, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    kbuild.build()
    K.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    inp = W.generate(wl, dev)
    T, H, d = wl.total_tokens, wl.heads, wl.head_dim
    B, Wd = wl.budget, wl.width
    ids = torch.empty((T, B), dtype=torch.int32, device=dev)
    toks = torch.empty((T, Wd), dtype=torch.int32, device=dev)
    ws = K.new_workspace(T, wl.num_seqs, H, d, K.KPOOL_BF16 if wl.dtype == "bf16" else K.KPOOL_F32, wl.kpool,
                         wl.index_topk, dev)
    # five events per timed step, recorded by the library around its four kernels
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for evs in step_events:
        for e in evs:
            e.record(stream)
    events = step_events[0]
    pairs = wl.causal_pairs()
    flops = FLOP_PER_PAIR_PER_HEAD_DIM * H * d * pairs

    def step(ev=None):
        K.kpool_select_ex(inp["q"], inp["k"], inp["w"], inp["cu_seqlens"], wl.kpool, wl.index_topk, wl.scale,
                          out_pool_ids=ids, out_token_ids=toks, workspace=ws, stream=stream, stage_events=ev)

    for _ in range(args.warmup):
        step(events)
    torch.cuda.synchronize()
    st = K.kpool_last_device_error(ws)
    if st != K.KPOOL_OK:
        raise K.KpoolError(st, "device")

    # ---- timed region: inputs resident in HBM (q alone is far larger than L2)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s_i in range(args.steps):
        step(step_events[s_i])
    t_end.record(stream)
    torch.cuda.synchronize()
    per_kernel = [[evs[i].elapsed_time(evs[i + 1]) for evs in step_events] for i in range(4)]
    barrier(world)
    clock_info = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    ms_step = max_over_ranks(ms_total / args.steps, world)
    st = K.kpool_last_device_error(ws)
    if st != K.KPOOL_OK:
        raise K.KpoolError(st, "device")
    value = world * pairs / (ms_step / 1e3)
    k_ms = [statistics.median(x) for x in per_kernel]  # per-kernel medians over the timed steps

    # ---- the gated pooling variant of step 1 (kpool_pool_keys_gated), timed on its own
    gg = torch.Generator(device=dev)
    gg.manual_seed(wl.seed + 101)
    gate = torch.randn((T, d), generator=gg, device=dev) * 2.0
    ape = torch.randn((wl.kpool, d), generator=gg, device=dev) * 0.25
    kp_g = torch.empty((T // wl.kpool, d), dtype=inp["k"].dtype, device=dev)
    gws = K.new_workspace(T, wl.num_seqs, 1, d, K.KPOOL_BF16 if wl.dtype == "bf16" else K.KPOOL_F32, wl.kpool, 0, dev)
    for _ in range(args.warmup):
        K.kpool_pool_keys_gated(inp["k"], gate, ape, inp["cu_seqlens"], wl.kpool, out=kp_g, workspace=gws,
                                stream=stream)
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ga.record(stream)
    for _ in range(args.steps):
        K.kpool_pool_keys_gated(inp["k"], gate, ape, inp["cu_seqlens"], wl.kpool, out=kp_g, workspace=gws,
                                stream=stream)
    gb.record(stream)
    torch.cuda.synchronize()
    gated_ms = ga.elapsed_time(gb) / args.steps  # plan + gated pooling
    del gate, kp_g, gws

    # a device-to-device copy moving the same number of bytes as the mean pooling (half read,
    # half written): what a transfer of this size reaches on this GPU, for context
    half = (T * d * 2 + wl.num_pools() * d * 2) // 2
    c_src = torch.empty(half, dtype=torch.uint8, device=dev)
    c_dst = torch.empty_like(c_src)
    c_ts = []
    for _ in range(args.warmup + 10):
        ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ca.record(stream)
        c_dst.copy_(c_src)
        cb.record(stream)
        torch.cuda.synchronize()
        c_ts.append(ca.elapsed_time(cb))
    copy_same_ms = statistics.median(c_ts[args.warmup:])
    del c_src, c_dst

    # ---- end to end through the C ABI with host buffers: every step copies its inputs
    # from pinned host memory and its pool and token ids back, pipelined the way a caller
    # would drive the library -- two device buffer sets; while step i computes on the main
    # stream, one copy stream downloads step i-1's results and then uploads step i+1's
    # inputs. Uploads and downloads share that stream on purpose: on this host, a download
    # running at the same time as an upload slows both several-fold, while one after the
    # other they take ~50 ms of a ~220 ms step.
    e2e = None
    if not args.no_e2e:
        h_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inp.items()}
        for k in h_in:
            h_in[k].copy_(inp[k])
        d_in = [inp, {k: torch.empty_like(v) for k, v in inp.items()}]
        d_ids = [ids, torch.empty_like(ids)]
        d_toks = [toks, torch.empty_like(toks)]
        h_ids = [torch.empty(ids.shape, dtype=ids.dtype, pin_memory=True) for _ in range(2)]
        h_toks = [torch.empty(toks.shape, dtype=toks.dtype, pin_memory=True) for _ in range(2)]
        bi = sum(v.numel() * v.element_size() for v in h_in.values())
        bo = h_ids[0].numel() * 4 + h_toks[0].numel() * 4
        up = torch.cuda.Stream()
        down = up  # one copy stream (see above)
        computed = [torch.cuda.Event(), torch.cuda.Event()]
        uploaded = [torch.cuda.Event(), torch.cuda.Event()]
        downloaded = [torch.cuda.Event(), torch.cuda.Event()]
        # timeline of the timed steps: upload, selection and download intervals on their own
        # streams (events on the stream each interval runs on)
        tl = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]

        def e2e_steps(n, marks=None):
            def download(j):
                b = j & 1
                ev = marks[j] if marks is not None else None
                up.wait_event(computed[b])
                with torch.cuda.stream(up):
                    if ev:
                        ev[4].record(up)
                    h_ids[b].copy_(d_ids[b], non_blocking=True)
                    h_toks[b].copy_(d_toks[b], non_blocking=True)
                    downloaded[b].record(up)
                    if ev:
                        ev[5].record(up)

            for i in range(n):
                b = i & 1
                ev = marks[i] if marks is not None else None
                # step i's inputs go into the buffers step i-2 read: the copy stream passed
                # step i-2's `computed` event before downloading its results
                with torch.cuda.stream(up):
                    if ev:
                        ev[0].record(up)
                    for k in h_in:
                        d_in[b][k].copy_(h_in[k], non_blocking=True)
                    uploaded[b].record(up)
                    if ev:
                        ev[1].record(up)
                stream.wait_event(uploaded[b])
                if i >= 2:
                    stream.wait_event(downloaded[b])  # step i-2's results have left these buffers
                if ev:
                    ev[2].record(stream)
                K.kpool_select_ex(d_in[b]["q"], d_in[b]["k"], d_in[b]["w"], d_in[b]["cu_seqlens"], wl.kpool,
                                  wl.index_topk, wl.scale, out_pool_ids=d_ids[b], out_token_ids=d_toks[b],
                                  workspace=ws, stream=stream)
                computed[b].record(stream)
                if ev:
                    ev[3].record(stream)
                if i >= 1:
                    download(i - 1)  # runs while step i computes
            download(n - 1)

        e2e_steps(2)
        torch.cuda.synchronize()
        # the same upload alone (nothing else on the GPU), to tell copy speed from overlap effects
        iso = []
        for _ in range(2):
            a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(up):
                a0.record(up)
                for k in h_in:
                    d_in[1][k].copy_(h_in[k], non_blocking=True)
                b0.record(up)
            torch.cuda.synchronize()
            iso.append(a0.elapsed_time(b0))
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_stream(stream)
        e2e_steps(args.steps, tl)
        stream.wait_stream(up)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(a.elapsed_time(b) / args.steps, world)
        med = lambda xs: statistics.median(xs) if xs else None  # noqa: E731
        timeline = {
            "upload_ms": med([e[0].elapsed_time(e[1]) for e in tl]),
            "select_ms": med([e[2].elapsed_time(e[3]) for e in tl]),
            "download_ms": med([e[4].elapsed_time(e[5]) for e in tl]),
            # time the selection stream sat idle between two selections (waiting on copies)
            "select_gap_ms": med([tl[i - 1][3].elapsed_time(tl[i][2]) for i in range(1, len(tl))]),
            "select_gap_total_ms": sum(tl[i - 1][3].elapsed_time(tl[i][2]) for i in range(1, len(tl))),
            "upload_max_ms": max(e[0].elapsed_time(e[1]) for e in tl),
            "upload_ms_by_step": [round(e[0].elapsed_time(e[1]), 2) for e in tl],
            "download_ms_by_step": [round(e[4].elapsed_time(e[5]), 2) for e in tl],
            "download_max_ms": max(e[4].elapsed_time(e[5]) for e in tl),
            "exposed_first_upload_ms": a.elapsed_time(tl[0][2]),
            "exposed_last_download_ms": tl[-1][3].elapsed_time(b),
            "select_alone_ms": ms_step,
            "upload_alone_ms": min(iso),
            "note": "medians over the timed steps; select_ms against select_alone_ms shows whether the selection "
                    "slows while copies run, select_gap_ms whether it waits on them"}
        e2e = {"value": world * pairs / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
               "pipelining": "2 buffer sets; one copy stream downloads step i-1 and uploads step i+1 while step i "
                             "computes",
               "timeline": timeline}
        st = K.kpool_last_device_error(ws)
        if st != K.KPOOL_OK:
            raise K.KpoolError(st, "device (end-to-end run)")
        del d_in, h_in, h_ids, h_toks

    peaks = measured_peaks()
    peak_burst = float(peaks["bf16_tflops"])
    peak_sust = float(peaks.get("bf16_tflops_sustained", peak_burst))
    k2_s = k_ms[2] / 1e3
    achieved = flops / k2_s / 1e12
    tc_src = os.path.join(ROOT, "sparse_attention_kpool_gb300", "csrc", "kpool_select_tc.cu")
    traffic = None
    if NCU_TRAFFIC["kernel_sha256"] == source_sha(tc_src) and NCU_TRAFFIC["workload"] == wl.name:
        traffic = NCU_TRAFFIC["bytes_per_launch"]
    hbm = float(peaks["hbm_gbs"])
    # q, w and k's pooled rows read once, pool ids written
    k2_bytes = T * H * d * 2 + T * H * 4 + wl.num_pools() * d * 2 + T * B * 4
    kp_bytes = wl.num_pools() * d * 2
    k1_bytes = T * d * 2 + kp_bytes
    k3_bytes = T * B * 4 + T * Wd * 4
    kg_bytes = T * d * 2 + T * d * 4 + wl.kpool * d * 4 + kp_bytes  # keys, fp32 gate scores, embedding in; pools out

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, world),
        "sec_per_selection": ms_step / 1e3,
        "scored_pairs_per_s": value,
        "pct_bf16_peak": 100.0 * achieved / peak_burst,
        "pct_bf16_peak_sustained": 100.0 * achieved / peak_sust,
        "kernel_ms": {"plan": k_ms[0], "pool": k_ms[1], "score_select": k_ms[2], "expand": k_ms[3]},
        "roofline": {"kernel": "select_tc_kernel (score+select)", "bound": "tensor", "achieved": achieved,
                     "peak": peak_burst, "unit": "TFLOP/s", "frac": achieved / peak_burst, "traffic": traffic,
                     "peak_kind": f"bf16 burst, {peaks['_source']}",
                     "frac_of_sustained": achieved / peak_sust,
                     "algorithmic_flop_per_launch": flops,
                     "algorithmic_bytes_per_launch": k2_bytes},
        "hbm_kernels": {
            "pool": {"bytes": k1_bytes, "GB/s": k1_bytes / (k_ms[1] / 1e3) / 1e9,
                     "frac": k1_bytes / (k_ms[1] / 1e3) / 1e9 / hbm,
                     "same_size_copy_GB/s": 2 * half / (copy_same_ms / 1e3) / 1e9},
            "expand": {"bytes": k3_bytes, "GB/s": k3_bytes / (k_ms[3] / 1e3) / 1e9,
                       "frac": k3_bytes / (k_ms[3] / 1e3) / 1e9 / hbm},
            "pool_gated": {"bytes": kg_bytes, "ms": gated_ms, "GB/s": kg_bytes / (gated_ms / 1e3) / 1e9,
                           "frac": kg_bytes / (gated_ms / 1e3) / 1e9 / hbm,
                           "note": "kpool_pool_keys_gated (plan + gated pooling), not part of the timed step"}},
        "clocks": clock_info,
        "gpu_launches": 4 * args.steps,
        "e2e": e2e,
    }
    if wl.name == "pages_512k":
        # the pages' own figure, context only (vs_baseline stays null): a different
        # implementation that scores the full query x pool rectangle, on another GPU
        line["pages_context"] = {
            "sec_per_selection": PAGES_SEC_512K, "hardware": "one B200 (as the pages state)",
            "work": "full query x pool rectangle (2x the causal pairs counted here)",
            "ratio_of_seconds": PAGES_SEC_512K / (ms_step / 1e3)}

    if wl.name == "pages_512k" and not args.no_decode:
        # the decode workload (16 rows against 262,144-token key caches) measured in the same
        # run, so its numbers come with the default bench line; its own oracle timing and
        # parity sample run only in its standalone run (--workload decode_262k)
        dec_args = argparse.Namespace(**vars(args))
        dec_args.steps, dec_args.warmup, dec_args.no_cpu = max(args.steps, 20), max(args.warmup, 5), True
        dec = rows_bench(dec_args, W.DECODE_262K, world, rank, emit=False)
        line["decode_262k"] = {k: dec[k] for k in ("metric", "value", "unit", "ms_per_step", "us_per_decode_step",
                                                   "us_per_decode_step_graph", "kernel_ms", "roofline", "clocks",
                                                   "config", "e2e", "steps", "warmup")}
    if wl.name == "pages_512k" and not args.no_index_scores:
        # the full index-score output on long_128k (2 GiB chunks), measured in the same run;
        # its oracle timing and parity sample run only standalone (--index-scores)
        sc_args = argparse.Namespace(**vars(args))
        sc_args.steps, sc_args.no_cpu = min(args.steps, 10), True
        isc = index_scores_bench(sc_args, W.LONG_128K, world, rank, emit=False)
        line["index_scores_long_128k"] = {k: isc[k] for k in ("metric", "value", "unit", "ms_per_step",
                                                              "kernel_ms", "roofline", "clocks", "config", "e2e",
                                                              "steps", "warmup")}
    if rank == 0 and not args.no_cpu:
        rows = pick_sample_rows(wl, args.cpu_sample_pairs, seed=7)
        res = oracle_sample(inp, wl, rows)
        cpu_value = res["pairs"] / res["seconds"]
        line["cpu_baseline"] = {
            "value": cpu_value, "unit": UNIT, "cores": res["threads"], "kind": "oracle",
            "sample": f"{len(rows)} uniform rows of {wl.name} ({res['pairs']:.3e} eligible pairs, "
                      f"{res['seconds']:.1f} s incl. pooling all keys); fp64 scores",
            "sec_per_selection_extrapolated": pairs / cpu_value}
        # the same rows double as a parity spot check of this run's output
        from tests import parity
        r = torch.as_tensor(rows, device=dev)
        sc_ids = ids[r].cpu().numpy()
        ok = True
        try:
            parity.compare_float(inp, wl, dict(res["out"], rows=rows, kp=res["kp"]), sc_ids, None,
                                 toks[r].cpu().numpy())
        except AssertionError as ex:
            ok = False
            line["parity_sample_error"] = str(ex)[:200]
        line["parity_sample"] = {"rows": int(len(rows)), "ok": ok}
        if wl.values == "integer":
            # rows of the sample where an exact tie straddles the budget cutoff (rank budget and
            # rank budget + 1 score the same, so the smaller-index rule decides): a one-slot-wider
            # oracle selection of the same rows
            from oracle import oracle as orc
            cu_h = inp["cu_seqlens"].cpu().numpy()
            wide = orc.select(parity.bits(inp["q"][r]), inp["w"][r].cpu().numpy(), res["kp"], cu_h, rows, wl.dtype,
                              wl.kpool, wl.index_topk + wl.kpool, wl.scale)
            line["cutoff_tie_rows"] = {"rows": int(len(parity.cutoff_tie_rows(wide, wl.budget))),
                                       "of_sampled": int(len(rows)),
                                       "with_more_eligible_than_budget": int((wide["eligible"] > wl.budget).sum())}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
