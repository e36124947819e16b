#!/usr/bin/env python
"""Benchmark of the DSA decode step on GB300: query-tokens/s of one pass of the whole hot path
(store this step's index keys -> indexer logits -> top-k -> sparse MLA), plus each stage's
achieved HBM bandwidth against its roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Defaults: N = 1, K = 20, W = 5, workload decode_b64_logu64k (64 requests, contexts log-uniform in
[4096, 65536], 1 query token each, top-k 2048, 128 MLA heads).  Under torchrun (N > 1) every rank
runs its own independent batch (seed offset by the rank) with no collective on the data path;
value = all ranks' query rows / the slowest rank's step time (weak scaling).

``--impl reference`` times the CPU oracle (the plain C definition of the path) on the host cores,
each step a bounded sample of the same workload; under torchrun only rank 0 runs it.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA decode query-tokens/s (indexer+top-k+sparse MLA); HBM GB/s vs roofline"
UNIT = "query-tokens/s"
DEFAULT_WORKLOAD = "decode_b64_logu64k"
L2_FLUSH_BYTES = 256 << 20
LAUNCHES_PER_STEP = 5       # store, logits, top-k, MLA split, MLA combine


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- algorithmic work

def algorithmic_work(wl):
    """Bytes (and FLOPs) each stage must move/compute at minimum, per step.
    indexer: 132 B per visible key per request (K read once per request) + 4 B per (row, key)
             logit written + q (bf16) and w (fp32) reads; 2*64*128 FLOP per (row, key).
    top-k:   4 B per (row, visible key) read + 4k B per row written.
    MLA:     per row: k * 1152 B gathered + q (H*576*2) + out (H*512*2) + idx (4k) + lse (4H);
             2 * H * k_valid * (576 + 512) FLOP.
    store:   per new token 256 B read + 132 B written + 8 B slot.
    indexer_c8: as indexer with 130 B per key (128 int8 codes + an fp16 scale)."""
    import numpy as np
    vis = wl.visible_lens().astype(np.int64)
    keys_per_req = wl.seq_lens.astype(np.int64)
    T, H, k = wl.T, wl.heads, wl.topk
    kvalid = np.minimum(vis, k)
    idx_b = int(keys_per_req.sum()) * 132 + int(vis.sum()) * 4 + T * 64 * 128 * 2 + T * 64 * 4
    idx_f = int(vis.sum()) * 2 * 64 * 128
    topk_b = int(vis.sum()) * 4 + T * k * 4
    mla_b = int(kvalid.sum()) * 1152 + T * H * 576 * 2 + T * H * 512 * 2 + T * k * 4 + T * H * 4
    mla_f = int(kvalid.sum()) * 2 * H * (576 + 512)
    store_b = T * (256 + 132 + 8)
    idx8_b = idx_b - int(keys_per_req.sum()) * 2
    return {"store": (store_b, 0), "indexer": (idx_b, idx_f), "topk": (topk_b, 0), "mla": (mla_b, mla_f),
            "indexer_c8": (idx8_b, idx_f)}


def compressed_device(c, db):
    """Device buffers of the compressed-KV stages: the FP8 index cache of the compressed keys, the
    compressed latent rows, their page table, sinks, the selection and the workspaces."""
    import numpy as np
    import torch
    from deepseek_sparse_attention_paged_gb300 import capi
    dev = db.device
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    pool = torch.zeros((c.num_pages, capi.INDEX_PAGE_BYTES), dtype=torch.uint8, device=dev)
    capi.dsa_store_index_k(bf(c.index_keys()), torch.from_numpy(c.slots()).to(dev), pool, db.dev_err)
    T, H = c.base.T, c.base.heads
    return {"pool": pool, "bt": torch.from_numpy(c.block_table).to(dev), "kv": bf(c.latent_pool()),
            "sinks": torch.from_numpy(c.sinks()).to(dev),
            "idx": torch.empty((T, c.topk), dtype=torch.int32, device=dev),
            "li_ws": torch.empty(capi.dsa_lightning_indexer_workspace_size(T, c.max_cmp_len), dtype=torch.uint8,
                                 device=dev),
            "attn_ws": torch.empty(max(16, capi.dsa_sparse_attn_swa_cmp_workspace_size(T, H, c.window, c.topk)),
                                   dtype=torch.uint8, device=dev),
            "out": torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((T, H), dtype=torch.float32, device=dev)}


def compressed_work(c):
    """Algorithmic bytes / FLOPs of the compressed-KV stages.
    dsv4_select: 132 B per compressed entry per request + 4 B per (row, visible entry) logit written
                 and read back by the top-k + the query and gates; 2*64*128 FLOP per (row, entry).
    dsv4_attn:   per row: (window keys + selected entries) * 1152 B + query, output, indices, lse;
                 2 * H * keys * (576 + 512) FLOP."""
    import numpy as np
    wl = c.base
    vis = wl.visible_lens().astype(np.int64)
    visc = vis // c.ratio
    T, H = wl.T, wl.heads
    sel_b = int(c.cmp_lens.astype(np.int64).sum()) * 132 + int(visc.sum()) * 8 + T * 64 * 128 * 2 + T * 64 * 4 \
        + T * c.topk * 4
    sel_f = int(visc.sum()) * 2 * 64 * 128
    keys = np.minimum(vis, c.window) + np.minimum(visc, c.topk)
    att_b = int(keys.sum()) * 1152 + T * H * 576 * 2 + T * H * 512 * 2 + T * c.topk * 4 + T * H * 4
    att_f = int(keys.sum()) * 2 * H * (576 + 512)
    return {"dsv4_select": (sel_b, sel_f), "dsv4_attn": (att_b, att_f)}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.sel = sel
        self.cmd = self._cmd(25)

    def _cmd(self, ms: int):
        return ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", str(ms)] + self.sel

    def _start(self):
        self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def __enter__(self):
        # sample every 25 ms (the timed region lasts tens of milliseconds); fall back to 100 ms if
        # this nvidia-smi gives nothing at that rate
        try:
            self._start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 2.0 and self.proc.poll() is None:
                time.sleep(0.02)
            if not self.lines:
                self.__exit__(None, None, None)
                self.cmd = self._cmd(100)
                self._start()
        except Exception:
            self.proc = None
        return self

    def wait_first_sample(self, timeout_s: float = 5.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout_s:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- profile traffic

def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "deepseek_sparse_attention_paged_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(stage, workload=DEFAULT_WORKLOAD):
    """DRAM bytes per launch from the committed ncu summary, only if the kernel source is unchanged
    and the summary is of this workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(stage)
    if not d or d.get("workload", DEFAULT_WORKLOAD) != workload:
        return None
    if d.get("source_hash") != kernel_source_hash(d["sources"]):
        return None
    return d.get("dram_bytes_per_launch_scaled", d.get("dram_bytes_per_launch"))


STAGE_SOURCES = {"store": ["store_index_k.cu"], "indexer": ["indexer_logits.cu"], "topk": ["topk.cu"],
                 "mla": ["sparse_mla.cu"]}
# tensor peak of each stage relative to the measured dense bf16 peak: the indexer contracts FP8
# operands (nominal dense FP8 : BF16 = 4.5 : 2.25 PFLOP/s), the attention bf16
STAGE_TENSOR_PEAK_RATIO = {"indexer": 2.0, "select": 2.0, "mla": 1.0, "dsv4_select": 2.0}
# per-tensor scales of the FP8 latent-cache stage (~ max |N(0,1)| / 448 for the synthetic cache)
FP8_K_SCALE = 0.0125
FP8_Q_SCALE = 0.0125


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_sample_step(wl, rows, pools, rng_rows=None):
    """One decode step of the oracle for the given rows (their requests' index caches prebuilt):
    store the rows' new keys, score, select, attend.  Returns rows processed."""
    import numpy as np
    import oracle
    rows = np.asarray(rows, np.int64)
    cu = wl.cu_q
    new_ids = wl.new_token_ids()
    for r in rows:
        b = int(np.searchsorted(cu, r, side="right") - 1)
        pool = pools[b]
        oracle.store_index_k(wl.index_keys()[new_ids[r:r + 1]], wl.token_slots()[new_ids[r:r + 1]], pool)
        lg = oracle.indexer_logits(wl.index_q(), wl.weights(), pool, wl.block_table, wl.seq_lens, wl.cu_q,
                                   np.array([r]), wl.max_seq_len)
        idx = oracle.topk(lg, wl.seq_lens, wl.cu_q, np.array([r]), wl.topk)
        full = np.full((wl.T, wl.topk), -1, np.int32)
        full[r] = idx[0]
        oracle.sparse_mla(wl.mla_q(), wl.latent_pool(), wl.block_table, wl.seq_lens, wl.cu_q, full, wl.scale,
                          np.array([r]))
    return len(rows)


def build_oracle_pools(wl, reqs):
    import numpy as np
    import oracle
    starts = np.concatenate([[0], np.cumsum(wl.seq_lens.astype(np.int64))])
    pools = {}
    for b in sorted(set(reqs)):
        pool = np.zeros((wl.num_pages, oracle.PAGE_BYTES), np.uint8)
        oracle.store_index_k(wl.index_keys()[starts[b]:starts[b + 1]], wl.token_slots()[starts[b]:starts[b + 1]],
                             pool)
        pools[b] = pool
    return pools


def sample_rows(wl, n):
    import numpy as np
    # rows evenly spaced over the batch (one per request for decode workloads)
    return np.unique(np.linspace(0, wl.T - 1, n).round().astype(np.int64))


def cpu_oracle_rate(wl, steps, rows_per_step, min_seconds=0.0):
    """Times the oracle on bounded samples: each step takes `rows_per_step` rows (evenly spaced over
    the batch, cycling) and runs the whole path for them; the index cache of their requests is
    built first, untimed (it is resident state, like the GPU's).  Runs `steps` steps, and more until
    `min_seconds` of timed CPU work have accumulated.  Returns (rows/s, cores, step times, rows)."""
    import numpy as np
    import oracle
    oracle.build()
    rows = sample_rows(wl, min(wl.T, 64))
    cu = wl.cu_q
    times, done, used = [], 0, []
    s = 0
    while s < steps or sum(times) < min_seconds:
        sel = [rows[(s * rows_per_step + i) % len(rows)] for i in range(rows_per_step)]
        reqs = [int(np.searchsorted(cu, r, side="right") - 1) for r in sel]
        pools = build_oracle_pools(wl, reqs)
        t0 = time.perf_counter()
        done += oracle_sample_step(wl, sel, pools)
        times.append(time.perf_counter() - t0)
        used.extend(int(r) for r in sel)
        del pools
        s += 1
    return done / sum(times), oracle.num_threads(), times, used


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from deepseek_sparse_attention_paged_gb300 import workloads
    wl = workloads.make(args.workload)
    rows_per_step = 1
    _, cores, _, _ = cpu_oracle_rate(wl, args.warmup, rows_per_step) if args.warmup > 0 else (0, 0, 0, 0)
    rate, cores, times, rows = cpu_oracle_rate(wl, args.steps, rows_per_step)
    ms = 1000.0 * sum(times) / max(1, len(times))
    sample = (f"{rows_per_step} query row per step (rows evenly spaced over the {wl.T}-row batch, each with its "
              f"full context: store its key, logits over its visible keys, top-{wl.topk}, {wl.heads}-head sparse "
              f"MLA); index caches of the sampled requests prebuilt untimed")
    line = {"metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(wl),
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def workload_config(wl):
    import numpy as np
    return {"workload": wl.name, "batch": wl.B, "query_rows": wl.T,
            "context_min": int(wl.seq_lens.min()), "context_max": int(wl.seq_lens.max()),
            "context_total": int(wl.seq_lens.astype(np.int64).sum()), "q_per_request": int(wl.max_q_len),
            "topk": wl.topk, "mla_heads": wl.heads, "index_heads": 64, "index_dim": 128, "page_size": 64,
            "index_pool_pages": wl.num_pages, "seed": wl.seed,
            "l2": "flushed between timed steps (256 MiB write, then 256 MiB read of another buffer; untimed)",
            "timing": "per timed iteration one replay of a CUDA graph holding the L2 flush, a timing event, "
                      "the step's kernels and a second timing event (events recorded by the graph, so the "
                      "graph's launch latency and the flush are outside the measured interval)"}


def capture(fn, stream):
    """CUDA graph of fn() on `stream`; returns (graph, kernels captured)."""
    import torch
    from deepseek_sparse_attention_paged_gb300 import capi
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the path outside capture
        torch.cuda.synchronize()
        n0 = capi.launch_count()
        with torch.cuda.graph(g, stream=stream):
            fn()
        n = capi.launch_count() - n0
    torch.cuda.synchronize()
    return g, n


class TimedGraph:
    """One CUDA graph per measured unit: an L2 flush (a 256 MiB write, then a 256 MiB read so that
    the written lines are back in HBM), then a timing event, the unit's kernels, a second timing
    event.  The events are recorded by the graph itself (external event nodes), so a replay's
    elapsed time is the device time of the kernels alone: neither the flush nor the graph's launch
    latency is inside it.  Where torch cannot record events inside a graph, the events are recorded
    around the replay instead (launch latency then included)."""

    _read = None   # the flush's read buffer, shared by every instance

    def __init__(self, fn, stream, flush):
        import torch
        from deepseek_sparse_attention_paged_gb300 import capi
        self.stream, self.flush = stream, flush
        # a second buffer read after the flush write: the write's dirty lines are written back to HBM
        # before the timed interval starts instead of during it
        if TimedGraph._read is None or TimedGraph._read.numel() != flush.numel():
            TimedGraph._read = torch.ones_like(flush)
        self.flush_read = TimedGraph._read
        try:
            self.a = torch.cuda.Event(enable_timing=True, external=True)
            self.b = torch.cuda.Event(enable_timing=True, external=True)
            self.inside = True
        except TypeError:
            self.a = torch.cuda.Event(enable_timing=True)
            self.b = torch.cuda.Event(enable_timing=True)
            self.inside = False
        self.g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()  # warm the path outside capture
            torch.cuda.synchronize()
            n0 = capi.launch_count()
            with torch.cuda.graph(self.g, stream=stream):
                if self.inside:
                    flush.fill_(1.0)
                    self.sink = self.flush_read.amax()
                    self.a.record(stream)
                fn()
                if self.inside:
                    self.b.record(stream)
            self.kernels = capi.launch_count() - n0
        torch.cuda.synchronize()

    def time(self, iters):
        """Per-replay device time (ms) of the unit's kernels, L2 flushed before each."""
        import torch
        out = []
        with torch.cuda.stream(self.stream):
            for _ in range(iters):
                if not self.inside:
                    self.flush.fill_(1.0)
                    self.a.record(self.stream)
                self.g.replay()
                if not self.inside:
                    self.b.record(self.stream)
                self.b.synchronize()
                out.append(self.a.elapsed_time(self.b))
        return out


def time_graph(g, stream, iters, flush):
    """Per-iteration CUDA-event time (ms) of one replay; L2 flushed before each, untimed."""
    import torch
    pairs = []
    with torch.cuda.stream(stream):
        for _ in range(iters):
            flush.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            pairs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in pairs]


def run_gpu(args):
    import numpy as np
    import torch
    from deepseek_sparse_attention_paged_gb300 import capi, workloads
    from deepseek_sparse_attention_paged_gb300.build import build
    from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    if rank == 0:
        build()
    if pg is not None:
        pg.barrier()
    capi.load()

    from deepseek_sparse_attention_paged_gb300 import distributed as D
    wl = D.rank_workload(args.workload, rank)   # every rank its own batch of the same shape
    db = DeviceBatch(wl, c8=True)   # the int8 index cache too, for its stage line
    stream = torch.cuda.Stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    step_graph = TimedGraph(lambda: db.step(), stream, flush)
    step_kernels = step_graph.kernels
    stage_graphs = {
        "store": TimedGraph(lambda: db.store_new_keys(), stream, flush),
        "indexer": TimedGraph(lambda: db.indexer_stage(), stream, flush),
        "topk": TimedGraph(lambda: db.topk_stage(), stream, flush),
        "select": TimedGraph(lambda: db.select(), stream, flush),
        "mla": TimedGraph(lambda: db.sparse_mla(), stream, flush),
    }
    # the FP8 latent-cache variant of the attention on the same selections (cache quantised on the
    # device by dsa_store_latent_fp8, per-tensor scales; timed as a stage of its own)
    kv8 = torch.empty((wl.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
    capi.dsa_store_latent_fp8(db.kv_pool.view(-1, 576), torch.arange(wl.num_pages * 64, device="cuda"), FP8_K_SCALE,
                              kv8)
    out8 = torch.empty_like(db.out)
    lse8 = torch.empty_like(db.lse)
    stage_graphs["mla_fp8"] = TimedGraph(
        lambda: capi.dsa_sparse_mla_decode_fp8(db.mla_q, FP8_Q_SCALE, kv8, FP8_K_SCALE, db.block_table, db.seq_lens,
                                               db.cu_q, db.idx, wl.scale, out8, db.mla_ws, lse=lse8,
                                               dev_err=db.dev_err), stream, flush)
    # the int8 ("c8") index-cache variant of the indexer logits over the same keys
    stage_graphs["indexer_c8"] = TimedGraph(lambda: db.indexer_c8_stage(), stream, flush)
    # the compressed-KV (ratio 4) layers: the one-call indexer over compressed keys, then the attention
    # over a 128-token window plus the selected compressed entries with per-head sinks
    cmp = workloads.make_compressed(wl)
    cmp_dev = compressed_device(cmp, db)
    capi.dsa_lightning_indexer(db.index_q, db.weights, cmp_dev["pool"], cmp_dev["bt"], db.seq_lens, db.cu_q,
                               cmp.max_cmp_len, wl.max_q_len, cmp.topk, cmp_dev["idx"], cmp_dev["li_ws"],
                               flags=capi.DSA_KEYS_CMP4, dev_err=db.dev_err)
    stage_graphs["dsv4_select"] = TimedGraph(
        lambda: capi.dsa_lightning_indexer(db.index_q, db.weights, cmp_dev["pool"], cmp_dev["bt"], db.seq_lens,
                                           db.cu_q, cmp.max_cmp_len, wl.max_q_len, cmp.topk, cmp_dev["idx"],
                                           cmp_dev["li_ws"], flags=capi.DSA_KEYS_CMP4, dev_err=db.dev_err),
        stream, flush)
    stage_graphs["dsv4_attn"] = TimedGraph(
        lambda: capi.dsa_sparse_attn_swa_cmp(db.mla_q, db.kv_pool, db.block_table, cmp_dev["kv"], cmp_dev["bt"],
                                             db.seq_lens, db.cu_q, cmp_dev["idx"], cmp.window, cmp.ratio,
                                             cmp_dev["sinks"], wl.scale, cmp_dev["out"], workspace=cmp_dev["attn_ws"],
                                             lse=cmp_dev["lse"], dev_err=db.dev_err), stream, flush)
    st, word = db.device_error()
    if st != 0:
        raise RuntimeError(f"device error word {word} after warm-up")

    clk = ClockSampler(local).__enter__()   # samples from warm-up through the e2e run
    clk.wait_first_sample()
    # warm-up steps (untimed)
    step_graph.time(args.warmup)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    step_ms = step_graph.time(args.steps)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    # stage breakdown (each stage alone in its own graph, same flush discipline), outside the K steps
    stage_iters = max(3, args.steps // 2)
    stage_ms = {k: g.time(stage_iters) for k, g in stage_graphs.items()}
    timed_launches = step_kernels * args.steps
    mean_step = D.max_over_ranks(sum(step_ms) / len(step_ms), device=torch.device("cuda", local))
    value = D.aggregate_rate(wl.T, world, mean_step)

    # e2e: same step through the public API with host buffers (pinned), copies inside the timing
    e2e = run_e2e(db, stream, args, flush)
    clk.__exit__(None, None, None)
    prologues = run_prologues(wl, stream, flush, stage_iters) if rank == 0 else None
    projections = run_projections(stream, flush, stage_iters) if rank == 0 else None

    if rank != 0:
        return
    hbm, bf16, peak_kind = measured_peaks()
    work = algorithmic_work(wl)
    work["select"] = tuple(a + b for a, b in zip(work["indexer"], work["topk"]))
    mb, mf = work["mla"]
    work["mla_fp8"] = (mb - int(np.minimum(wl.visible_lens(), wl.topk).sum()) * 576, mf)   # 576 B rows, not 1152
    work.update(compressed_work(cmp))
    stages = {}
    for k, ms_list in stage_ms.items():
        ms = sum(ms_list) / len(ms_list)
        b, f = work[k]
        tc = STAGE_TENSOR_PEAK_RATIO.get(k, 1.0) * bf16      # the stage's own operand type
        t_hbm, t_tc = b / (hbm * 1e9), f / (tc * 1e12)
        stages[k] = {"ms": ms, "algorithmic_bytes": b, "flops": f, "gbs": b / (ms * 1e-3) / 1e9,
                     "hbm_frac": (b / (ms * 1e-3) / 1e9) / hbm,
                     "tflops": f / (ms * 1e-3) / 1e12, "tensor_peak_tflops": tc,
                     "tensor_frac": (f / (ms * 1e-3) / 1e12) / tc,
                     "bound": "tensor" if t_tc > t_hbm else "hbm",
                     "roofline_ms": max(t_hbm, t_tc) * 1e3, "roofline_frac": max(t_hbm, t_tc) * 1e3 / ms}
    dominant = max(("indexer", "mla"), key=lambda k: stages[k]["ms"])
    d = stages[dominant]
    src = "measured" if peak_kind == "measured" else "fallback"
    if d["bound"] == "hbm":
        roofline = {"bound": "hbm", "achieved": d["gbs"], "peak": hbm, "unit": "GB/s", "frac": d["gbs"] / hbm,
                    "traffic": recorded_traffic(dominant, wl.name), "kernel": dominant,
                    "peak_source": f"{src} hbm_gbs (MEASURED_PEAKS.json)" if src == "measured" else "fallback 6.8 TB/s"}
    else:
        roofline = {"bound": "tensor", "achieved": d["tflops"], "peak": d["tensor_peak_tflops"], "unit": "TFLOP/s",
                    "frac": d["tensor_frac"], "traffic": recorded_traffic(dominant, wl.name), "kernel": dominant,
                    "peak_source": (f"{src} bf16_tflops (MEASURED_PEAKS.json, burst)"
                                    + (" x 2, the nominal FP8 : BF16 dense ratio" if
                                       STAGE_TENSOR_PEAK_RATIO.get(dominant, 1.0) == 2.0 else ""))}
    # CPU oracle baseline on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, cores, times, rows = cpu_oracle_rate(wl, 8, 1, min_seconds=10.0)
        # the same oracle on one host thread (a few rows)
        import oracle
        oracle.set_num_threads(1)
        rate1, _, times1, rows1 = cpu_oracle_rate(wl, 2, 1)
        oracle.set_num_threads(cores)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "single_thread": {"value": rate1, "rows": len(rows1), "seconds": sum(times1)},
               "sample": f"{len(rows)} query rows of the same batch (rows evenly spaced, cycling), one per step, "
                         f"each with its full context (store its key, logits over its visible keys, "
                         f"top-{wl.topk}, {wl.heads}-head sparse MLA); {sum(times):.1f} s of timed CPU work; "
                         f"the sampled requests' index caches built untimed"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8e4m3+bf16", "data": "synthetic", "config": workload_config(wl),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": timed_launches, "kernels_per_step": step_kernels,
            "clocks": clk.summary(), "stages": stages, "wall_s_timed_region": t_wall}
    hbm_peak = hbm
    for v in prologues.values():
        v["hbm_frac"] = v["gbs"] / hbm_peak
    line["indexer_prologues"] = prologues
    for v in projections.values():
        v["hbm_frac"] = v["gbs"] / hbm_peak
        v["tensor_frac"] = v["tflops"] / bf16
    line["mla_projections"] = projections
    print(json.dumps(line), flush=True)


def run_prologues(wl, stream, flush, iters):
    """Time the indexer prologue calls (key norm + rotary + rotate/quantise/store, and the query
    rotary embedding) at the decode shape of `wl` (its new keys, its query rows) and at a bulk,
    HBM-bound shape (a 131072-token prompt: keys at positions 0 .. 131071; 8192 query rows), each
    call alone in a CUDA graph, L2 flushed before every replay.  Algorithmic bytes: key prologue
    256 (raw key) + 256 (cos/sin row) + 16 (position, slot) read + 132 written per token; query
    rotary 64 x 256 read + 64 x 256 written + 256 + 8 read per row."""
    import numpy as np
    import torch
    from deepseek_sparse_attention_paged_gb300 import capi
    g = torch.Generator().manual_seed(wl.seed + 77)
    max_pos = 163840
    inv = 10000.0 ** (-torch.arange(0, 64, 2, dtype=torch.float64) / 64.0)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    cos_sin = torch.cat([ang.cos(), ang.sin()], dim=1).float().cuda()
    w = (1.0 + 0.1 * torch.randn(128, generator=g)).float().cuda()
    b = (0.1 * torch.randn(128, generator=g)).float().cuda()
    out = {}

    def key_case(n, positions, pages):
        k = torch.randn(n, 128, generator=g).to(torch.bfloat16).cuda()
        slots = torch.randperm(pages * 64, generator=g)[:n].cuda()
        pool = torch.zeros(pages, capi.INDEX_PAGE_BYTES, dtype=torch.uint8, device="cuda")
        pos = positions.cuda()
        tg = TimedGraph(lambda: capi.dsa_store_index_k_prologue(k, w, b, 1e-6, cos_sin, pos, slots, pool), stream, flush)
        ms = sum(tg.time(iters)) / iters
        by = n * (256 + 256 + 16 + 132)
        return {"tokens": n, "us": ms * 1e3, "algorithmic_bytes": by, "gbs": by / (ms * 1e-3) / 1e9}

    def q_case(T):
        q = torch.randn(T, 64, 128, generator=g).to(torch.bfloat16).cuda()
        qo = torch.empty_like(q)
        pos = torch.randint(0, max_pos, (T,), generator=g).cuda()
        tg = TimedGraph(lambda: capi.dsa_indexer_rope_q(q, cos_sin, pos, qo), stream, flush)
        ms = sum(tg.time(iters)) / iters
        by = T * (64 * 256 * 2 + 256 + 8)
        return {"rows": T, "us": ms * 1e3, "algorithmic_bytes": by, "gbs": by / (ms * 1e-3) / 1e9}

    new_pos = torch.from_numpy((wl.seq_lens.astype(np.int64) - 1) % max_pos)
    out["store_prologue_decode"] = key_case(wl.B, new_pos, max(1, (wl.B + 63) // 64) * 4)
    out["store_prologue_bulk"] = key_case(131072, torch.arange(131072), 131072 // 64)
    out["rope_q_decode"] = q_case(wl.T)
    out["rope_q_bulk"] = q_case(8192)
    return out


def run_projections(stream, flush, iters, heads=128):
    """Time the per-head projections around the absorbed attention (dsa_mla_absorb_q,
    dsa_mla_v_up) at a decode shape (64 rows) and a prefill-chunk shape (4096 rows), 128 heads,
    each call alone in a CUDA graph, L2 flushed before every replay.  Algorithmic work per call:
    the weights (heads x 128 x 512 bf16) read once, the input and output rows read / written once;
    2 x rows x heads x 128 x 512 FLOP."""
    import math
    import torch
    from deepseek_sparse_attention_paged_gb300 import capi
    g = torch.Generator().manual_seed(91)
    w_uk_t = (torch.randn(heads, 128, 512, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
    w_uv = (torch.randn(heads, 512, 128, generator=g) / math.sqrt(512)).to(torch.bfloat16).cuda()
    out = {}
    for T in (64, 4096):
        q = torch.randn(T, heads, 192, generator=g).to(torch.bfloat16).cuda()
        mla_q = torch.empty(T, heads, 576, dtype=torch.bfloat16, device="cuda")
        o = torch.randn(T, heads, 512, generator=g).to(torch.bfloat16).cuda()
        y = torch.empty(T, heads * 128, dtype=torch.bfloat16, device="cuda")
        flop = 2 * T * heads * 128 * 512
        wbytes = heads * 128 * 512 * 2
        for name, fn, by in (("absorb", lambda: capi.dsa_mla_absorb_q(q[..., :128], w_uk_t, mla_q[..., :512]),
                              wbytes + T * heads * (128 + 512) * 2),
                             ("v_up", lambda: capi.dsa_mla_v_up(o, w_uv, y.view(T, heads, 128)),
                              wbytes + T * heads * (512 + 128) * 2)):
            tg = TimedGraph(fn, stream, flush)
            ms = sum(tg.time(iters)) / iters
            out[f"{name}_T{T}"] = {"rows": T, "heads": heads, "us": ms * 1e3, "algorithmic_bytes": by, "flops": flop,
                                   "gbs": by / (ms * 1e-3) / 1e9, "tflops": flop / (ms * 1e-3) / 1e12}
    return out


def run_e2e(db, stream, args, flush):
    """End to end through the library's public API, with the step's inputs coming from and its
    outputs going to pinned host memory every step (one packed block each way):
      * value: DeviceBatch.run_io(), K steps back to back, the copies of step i +/- 1 overlapping
        the compute of step i (two device I/O sets); every step touches ~375 MB of index / latent
        cache, more than the 129 MB L2, so consecutive steps do not run from L2;
      * serial: DeviceBatch.step_io(), one step at a time (copies, four calls, copies as one CUDA
        graph), L2 flushed before each."""
    import torch
    wl = db.wl
    dev_in, dev_out = db.io_buffers()
    host_in = dev_in.cpu().pin_memory()
    host_outs = [torch.empty_like(dev_out, device="cpu").pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in db.io_inputs())
    d2h = sum(t.numel() * t.element_size() for t in db.io_outputs())
    K, W = args.steps, max(1, args.warmup)

    # pipelined stream of steps
    db.run_io([host_in] * W, [host_outs[i & 1] for i in range(W)], stream=stream)
    torch.cuda.synchronize()
    flush.fill_(1)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    db.run_io([host_in] * K, [host_outs[i & 1] for i in range(K)], stream=stream)
    b.record(stream)
    b.synchronize()
    ms_pipe = a.elapsed_time(b) / K

    # one step at a time
    for _ in range(W):
        db.step_io([host_in], [host_outs[0]], stream=stream)
    torch.cuda.synchronize()
    times = []
    for _ in range(K):
        flush.fill_(1)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        db.step_io([host_in], [host_outs[0]], stream=stream)
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms_serial = sum(times) / len(times)
    return {"value": wl.T / (ms_pipe / 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms_pipe,
            "api": "DeviceBatch.run_io(): per step the inputs as one packed block from pinned host memory, the "
                   "four C-ABI calls (one CUDA graph), the outputs as one packed block back to pinned host "
                   "memory; the copies of neighbouring steps overlap the compute on their own streams",
            "l2": "steps back to back; each touches ~375 MB of cache, more than the 129 MB L2",
            "serial": {"value": wl.T / (ms_serial / 1000.0), "ms_per_step": ms_serial,
                       "api": "DeviceBatch.step_io(), one step at a time, L2 flushed before each"}}


def run_profile(args):
    """Launches one stage (or the whole step) warmup + steps times with no timing, for a profiler.
    Only what the stage needs is put on the device (the latent cache only for `mla` / `step`)."""
    import torch
    from deepseek_sparse_attention_paged_gb300 import capi, workloads
    from deepseek_sparse_attention_paged_gb300.build import build
    from deepseek_sparse_attention_paged_gb300.pipeline import DeviceBatch
    build()
    capi.load()
    wl = workloads.make(args.workload)
    if args.profile in ("absorb", "v_up", "absorb4k"):
        # the shapes of run_projections: 64 rows (4096 for absorb4k), 128 heads
        import math
        g = torch.Generator().manual_seed(91)
        T, H = (4096 if args.profile == "absorb4k" else 64), 128
        if args.profile in ("absorb", "absorb4k"):
            w = (torch.randn(H, 128, 512, generator=g) / math.sqrt(128)).to(torch.bfloat16).cuda()
            q = torch.randn(T, H, 192, generator=g).to(torch.bfloat16).cuda()
            mla_q = torch.empty(T, H, 576, dtype=torch.bfloat16, device="cuda")
            fn = lambda: capi.dsa_mla_absorb_q(q[..., :128], w, mla_q[..., :512])
        else:
            w = (torch.randn(H, 512, 128, generator=g) / math.sqrt(512)).to(torch.bfloat16).cuda()
            o = torch.randn(T, H, 512, generator=g).to(torch.bfloat16).cuda()
            y = torch.empty(T, H * 128, dtype=torch.bfloat16, device="cuda")
            fn = lambda: capi.dsa_mla_v_up(o, w, y.view(T, H, 128))
        for _ in range(args.warmup + args.steps):
            fn()
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))
        return
    if args.profile in ("prologue", "rope_q"):
        # the bulk shapes of run_prologues: a 131072-token prompt's keys, 8192 query rows
        g = torch.Generator().manual_seed(wl.seed + 77)
        max_pos = 163840
        inv = 10000.0 ** (-torch.arange(0, 64, 2, dtype=torch.float64) / 64.0)
        ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
        cos_sin = torch.cat([ang.cos(), ang.sin()], dim=1).float().cuda()
        if args.profile == "prologue":
            n = 131072
            k = torch.randn(n, 128, generator=g).to(torch.bfloat16).cuda()
            w = (1.0 + 0.1 * torch.randn(128, generator=g)).float().cuda()
            b = (0.1 * torch.randn(128, generator=g)).float().cuda()
            slots = torch.randperm(n, generator=g).cuda()
            pos = torch.arange(n).cuda()
            pool = torch.zeros(n // 64, capi.INDEX_PAGE_BYTES, dtype=torch.uint8, device="cuda")
            fn = lambda: capi.dsa_store_index_k_prologue(k, w, b, 1e-6, cos_sin, pos, slots, pool)
        else:
            q = torch.randn(8192, 64, 128, generator=g).to(torch.bfloat16).cuda()
            qo = torch.empty_like(q)
            pos = torch.randint(0, max_pos, (8192,), generator=g).cuda()
            fn = lambda: capi.dsa_indexer_rope_q(q, cos_sin, pos, qo)
        for _ in range(args.warmup + args.steps):
            fn()
        torch.cuda.synchronize()
        print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))
        return
    need_latent = args.profile in ("mla", "step", "mla_fp8", "dsv4")
    db = DeviceBatch(wl, with_latent=need_latent, c8=args.profile == "indexer_c8")
    if args.profile in ("topk", "mla", "mla_fp8"):
        db.select()
    if args.profile == "dsv4":
        # the compressed-KV layers: the one-call indexer over compressed keys, then the attention
        cmp = workloads.make_compressed(wl)
        cd = compressed_device(cmp, db)

        def fn():
            capi.dsa_lightning_indexer(db.index_q, db.weights, cd["pool"], cd["bt"], db.seq_lens, db.cu_q,
                                       cmp.max_cmp_len, wl.max_q_len, cmp.topk, cd["idx"], cd["li_ws"],
                                       flags=capi.DSA_KEYS_CMP4, dev_err=db.dev_err)
            capi.dsa_sparse_attn_swa_cmp(db.mla_q, db.kv_pool, db.block_table, cd["kv"], cd["bt"], db.seq_lens,
                                         db.cu_q, cd["idx"], cmp.window, cmp.ratio, cd["sinks"], wl.scale, cd["out"],
                                         workspace=cd["attn_ws"], lse=cd["lse"], dev_err=db.dev_err)
    elif args.profile == "mla_fp8":
        # the FP8 latent cache of the same rows; the bf16 cache is dropped once it is quantised
        kv8 = torch.empty((wl.num_pages, 64, 576), dtype=torch.uint8, device="cuda")
        capi.dsa_store_latent_fp8(db.kv_pool.view(-1, 576), torch.arange(wl.num_pages * 64, device="cuda"),
                                  FP8_K_SCALE, kv8)
        torch.cuda.synchronize()
        db.kv_pool = None
        torch.cuda.empty_cache()
        out8, lse8 = torch.empty_like(db.out), torch.empty_like(db.lse)
        fn = lambda: capi.dsa_sparse_mla_decode_fp8(db.mla_q, FP8_Q_SCALE, kv8, FP8_K_SCALE, db.block_table,
                                                    db.seq_lens, db.cu_q, db.idx, wl.scale, out8, db.mla_ws,
                                                    lse=lse8, dev_err=db.dev_err)
    else:
        fn = {"store": db.store_new_keys, "indexer": db.indexer_stage, "topk": db.topk_stage,
              "mla": db.sparse_mla, "step": db.step, "indexer_c8": db.indexer_c8_stage}[args.profile]
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    st, word = db.device_error()
    print(json.dumps({"profile": args.profile, "workload": wl.name, "launches": args.warmup + args.steps,
                      "device_error": word}))
    if st != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--profile", choices=["store", "indexer", "topk", "mla", "step", "indexer_c8", "mla_fp8", "dsv4",
                                          "prologue", "rope_q", "absorb",
                                          "v_up", "absorb4k"],
                    default=None,
                    help="launch one stage warmup+steps times without timing (for ncu) and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.profile is not None:
        run_profile(args)
        return
    if args.warmup < 3 and args.impl == "native":
        print("note: warm-up raised to 3 (minimum)", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
