"""Benchmark of one hybrid-compressed-attention layer on GB300.

Headline workload: c4a decode, B=32 sequences of 32768 context tokens, one new token and
one query per sequence at position 32768. One step = one pass of the layer over the
batch: insert the new tokens (compressor + window + residual), indexer scores + top-512,
attention over the selected entries and the 128-token window with inverse RoPE.
Secondary (reported alongside): chunked prefill of 8192 tokens after 122880 cached ones,
with prefill attention TFLOP/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload (decode shards by
sequence; there is no data-path collective); rank 0 prints one JSON line.
--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import contextlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "c4a decode queries/s + HBM GB/s at B=32x32k; prefill attn TFLOP/s"
UNIT = "queries/s"
B, L = 32, 32768
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ algorithmic work
def decode_bytes_per_query(n_vis: int, k: int, swa: int, D: int = 512, H: int = 64,
                           H_I: int = 64, d_I: int = 128, idx_fp4: bool = False) -> dict:
    """Bytes one decode query must move at least (fp8 rows + fp32 row scale; the indexer
    rows packed fp4 + fp32 row scale with idx_fp4)."""
    parts = {
        "indexer_keys": n_vis * ((d_I // 2 if idx_fp4 else d_I) + 4),
        "selected_rows": k * (D + 4),
        "window_rows": swa * (D + 4),
        "q_and_out": 2 * H * D * 2,
        "q_idx_and_w": H_I * d_I * 2 + H_I * 4,
        "topk_ids": 2 * k * 4,
        "block_tables": 1024,
        "insert": 2 * (2 * D + 2 * d_I) * 2 + (D + 4),   # new token in, residual + window out
    }
    parts["total"] = sum(parts.values())
    return parts


def index_bytes_per_query(n_vis: int, k: int, H_I: int = 64, d_I: int = 128,
                          idx_fp4: bool = False) -> int:
    return n_vis * ((d_I // 2 if idx_fp4 else d_I) + 4) + H_I * d_I * 2 + H_I * 4 + k * 4


def attn_bytes_per_query(k: int, swa: int, H: int = 64, D: int = 512) -> int:
    """Selected and window rows (fp8 codes + fp32 scale), their ids, the query and the output."""
    return (k + swa) * (D + 4) + k * 4 + 2 * H * D * 2


def compress_bytes_per_token(D: int = 512, d_I: int = 128, S: int = 4, c4a: bool = True) -> int:
    """Bytes the insert must move per new token: read kv, s (and ik, is) in bf16, write the
    token's window row (fp8 codes + fp32 scale) and 1/S of an entry (attention row, and the
    indexer row for c4a); the residual rows of the last window are left out (per call)."""
    read = (2 * D + (2 * d_I if c4a else 0)) * 2
    entry = (D + 4) + ((d_I + 4) if c4a else 0)
    return read + (D + 4) + entry // S


def c128a_bytes_per_query(n_vis: int, swa: int, D: int = 512, H: int = 64) -> dict:
    """Dense c128a decode: every visible entry and window row (fp8 + scale), the query and
    the output, the sequence's block-table row (one int32 per 2-entry block) and the insert."""
    parts = {
        "entry_rows": n_vis * (D + 4),
        "window_rows": swa * (D + 4),
        "q_and_out": 2 * H * D * 2,
        "block_table": ((n_vis + 1) // 2) * 4,
        "insert": 2 * (2 * D) * 2 + (D + 4),     # new token in, residual + window out
    }
    parts["total"] = sum(parts.values())
    return parts


def mixed_bytes(lens, k: int = 512, swa: int = 128) -> dict:
    """Exact algorithmic bytes of one mixed decode step from the drawn lengths: the c4a layer
    (indexer keys of every visible entry, top-k + window rows, query/out, indexer query) and
    the c128a layer (every visible entry + window rows, query/out)."""
    c4a = c128 = 0
    for L in lens:
        n4 = max(0, (L - 8) // 4 + 1)
        n128 = max(0, (L - 128) // 128 + 1)
        c4a += decode_bytes_per_query(n4, min(k, n4), swa)["total"]
        c128 += c128a_bytes_per_query(n128, swa)["total"]
    return {"c4a_layer": c4a, "c128a_layer": c128, "total": c4a + c128}


def attn_flops_per_query(n_keys: int, H: int = 64, D: int = 512) -> float:
    return 4.0 * H * D * n_keys          # QK^T and PV, 2 flops per multiply-add


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", FALLBACK_HBM_GBS), d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), \
            d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


# ------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------ oracle arm
def oracle_sample_step(w, pools, sample):
    """The oracle's layer step for the sampled sequences: insert their new tokens (the
    other sequences get none), index + top-k, attention. Returns the queries processed."""
    from oracle import v4a_oracle as O
    h = w.layers[0]
    b, q = w.batch, w.queries
    sel = np.sort(np.asarray(sample))
    n_new = np.zeros(len(b.start), np.int64)
    n_new[sel] = b.cu[sel + 1] - b.cu[sel]
    cu = np.concatenate([[0], np.cumsum(n_new)])
    rows = np.concatenate([np.arange(b.cu[i], b.cu[i + 1]) for i in sel])
    O.compress_insert(h.spec, h.bias, h.gamma, h.ibias, pools, cu, b.start, b.kv[rows],
                      b.s[rows], b.ik[rows], b.is_[rows])
    top, _ = O.index_topk(h.spec, pools, q.seq[sel], q.pos[sel], q.q_idx[sel], q.w[sel],
                          h.spec.top_k)
    O.attention(h.spec, pools, q.seq[sel], q.pos[sel], q.q[sel], top)
    return len(sel)


def run_oracle(steps: int, warmup: int, n_sample: int, budget_s: float | None):
    """Time the oracle on host cores; each step is the layer step for n_sample queries."""
    import workloads as wl
    from oracle import v4a_oracle as O
    w = wl.c4a_decode(seed=1, B=B, L=L)
    h = w.layers[0]
    pools = O.Pools(h.spec, h.attn, h.idx, h.swa, h.state)
    rng = np.random.default_rng(0)
    samples = [rng.choice(B, n_sample, replace=False) for _ in range(steps + warmup)]
    for s in samples[:warmup]:
        oracle_sample_step(w, pools, s)
    t0 = time.perf_counter()
    done = 0
    n_steps = 0
    for s in samples[warmup:]:
        done += oracle_sample_step(w, pools, s)
        n_steps += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, dt, n_steps, done


def cpu_baseline_subprocess(n_sample: int, budget_s: float) -> dict:
    """The oracle in a fresh single-threaded process (BLAS pinned to one thread)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import bench, json; v, dt, n, q = bench.run_oracle(1000, 1, %d, %f); "
            "print(json.dumps([v, dt, n, q]))" % (n_sample, budget_s))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": "failed: " + r.stderr.strip().splitlines()[-1] if r.stderr else "failed"}
    v, dt, n, q = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%d layer steps of %d random sequences each (%d queries, %.1f s) of the "
                      "B=32 L=32768 c4a decode workload: insert + index/top-512 + attention "
                      "in numpy fp64" % (n, n_sample, q, dt)}


def reference_main(args, rank: int):
    if rank != 0:
        return
    n_sample = 2 if args.steps <= 500 else 1
    v, dt, n, q = run_oracle(args.steps, args.warmup, n_sample, None)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(n, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "c4a decode B=32 L=32768, oracle sample of %d sequences "
                                   "per step" % n_sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _blas_threads(),
                             "kind": "oracle",
                             "sample": "%d random sequences per step (insert + index/top-512 + "
                                       "attention), %d steps" % (n_sample, n)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _blas_threads() -> int:
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count() or 1


# -------------------------------------------------------------------------- GPU arm
def _dev(x, dt, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev, dt)


class DecodeReplica:
    """One copy of a decode workload's device state (pools + step inputs/outputs)."""

    def __init__(self, base_layer, w, dev, clone: bool, side: bool = False):
        import torch
        self.lay = base_layer.clone_pools() if clone else base_layer
        # decode: the insert runs on a side stream beside the indexer (Layer.step)
        self.side = torch.cuda.Stream(device=dev) if side else None
        b, q = w.batch, w.queries
        bf = torch.bfloat16
        opt = lambda x, dt: None if x is None else _dev(x, dt, dev)
        self.cu = _dev(b.cu, torch.int32, dev)
        self.start = _dev(b.start, torch.int64, dev)
        self.kv, self.s = _dev(b.kv, bf, dev), _dev(b.s, bf, dev)
        self.ik, self.is_ = opt(b.ik, bf), opt(b.is_, bf)
        self.q_seq, self.q_pos = _dev(q.seq, torch.int32, dev), _dev(q.pos, torch.int64, dev)
        self.q, self.q_idx = _dev(q.q, bf, dev), opt(q.q_idx, bf)
        self.w = opt(q.w, torch.float32)
        self.max_pos = int(q.pos.max())
        k = max(self.lay.top_k, 1)
        self.topk = torch.empty((len(q.pos), k), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)   # device error bits
        # query-norm weight and output of the fused insert + query RMSNorm call
        self.q_gamma = _dev(np.random.default_rng(7).normal(1.0, 0.1, self.q.shape[-1]),
                            torch.float32, dev)
        self.qn = torch.empty_like(self.q)

    def step(self):
        self.lay.step(self.cu, self.start, self.kv, self.s, self.ik, self.is_, self.q_seq,
                      self.q_pos, self.max_pos, self.q, self.q_idx, self.w, out=self.out,
                      dev_err=self.err, side_stream=self.side,
                      topk_out=self.topk if self.lay.top_k else None)

    def touched_bytes(self):
        n_vis = (self.max_pos - 8) // 4 + 1
        fp4 = self.lay.cfg.idx_format == 1
        return len(self.q) * decode_bytes_per_query(n_vis, self.lay.top_k, 128,
                                                    idx_fp4=fp4)["total"]


def chained_ms_per_step(step_fns, steps, warmup, stream):
    """Device time per step: one CUDA graph holds one step of every replica in turn (the
    replicas' steps linked by programmatic dependent launch, as a model's layers run in
    one graph), replayed; a tail graph of the first steps % n replicas makes the count
    exactly `steps`. Returns (ms per step, the graphs for reuse)."""
    import torch
    n = len(step_fns)
    for f in step_fns:
        f()
    torch.cuda.synchronize()

    def cap(fs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for f in fs:
                f()
        return g

    chain = cap(step_fns)
    tail = cap(step_fns[:steps % n]) if steps % n else None
    for _ in range(max(1, -(-warmup // n))):
        chain.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps // n):
        chain.replay()
    if tail is not None:
        tail.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def n_replicas(bytes_per_step: int, l2: int, fixed: int = 0) -> int:
    """Pool replicas so that the replicas' working set is at least 4x L2 (every step then
    reads its pools from HBM)."""
    return fixed or max(2, int(math.ceil(4.0 * l2 / bytes_per_step)))


def gpu_main(args, rank: int, world: int, local_rank: int):
    import torch
    import compressed_sparse_long_gb300 as v4a
    import workloads as wl
    from compressed_sparse_long_gb300.layer import Layer

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    v4a.library()
    hbm_peak, tf_peak, tf_sus, peak_src = peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or getattr(props, "l2_cache_size", 0) or (126 << 20)

    # profiling aids: one secondary workload alone
    if args.only == "prefill":
        print(json.dumps({"prefill": _prefill(dev, tf_peak, tf_sus)}), flush=True)
        return
    if args.only == "c128a":
        print(json.dumps({"c128a_decode": _c128a_decode(dev, args, l2, hbm_peak, tf_peak, rank,
                                                        world)}), flush=True)
        return
    if args.only == "mixed":
        print(json.dumps({"mixed_decode": _mixed_decode(dev, args, l2, hbm_peak, rank, world)}),
              flush=True)
        return
    if args.only == "compress":
        print(json.dumps({"compressor_aux": _compressor_aux(dev, hbm_peak)}), flush=True)
        return
    w = wl.c4a_decode(seed=rank_seed(rank), B=B, L=L)
    base = Layer.from_host(w.layers[0], dev)
    side = not args.serial_step
    r0 = DecodeReplica(base, w, dev, clone=False, side=side)
    per_step = r0.touched_bytes()
    n_rep = args.replicas or max(2, int(math.ceil(4.0 * l2 / per_step)))
    reps = [r0] + [DecodeReplica(base, w, dev, clone=True, side=side) for _ in range(n_rep - 1)]
    stream = torch.cuda.current_stream()

    # warm-up (also allocates the workspaces). The timed graphs chain the replicas' steps
    # the way a model's layers run back to back in one graph: one graph holds one step of
    # every replica (different batches and pools), consecutive steps linked by
    # programmatic dependent launch; a tail graph makes the count exactly --steps.
    for r in reps:
        r.step()
    torch.cuda.synchronize()

    def capture(rs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for r in rs:
                r.step()
        return g

    def run_steps(chain, tail, k):
        for _ in range(k // n_rep):
            chain.replay()
        if k % n_rep:
            tail[k % n_rep].replay()

    chain = capture(reps)
    tails = {args.steps % n_rep: capture(reps[:args.steps % n_rep])} if args.steps % n_rep else {}
    graphs = [capture([r]) for r in reps]          # one graph per step, reported beside
    torch.cuda.synchronize()
    # compress (1) + indexer scores (1) + top-k (1) + attention (1, or 2 with a separate
    # split merge), as the library plans the call
    _, attn_kernels = v4a.v4a_attn_plan(base.cfg, B, L, 512, False)
    launches_per_step = 3 + attn_kernels

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # load phase so the clock sampler sees the GPU busy, then the timed region
    with ClockSampler(local_rank) as clk:
        for i in range(-(-args.warmup // n_rep)):
            chain.replay()
        t_end = time.perf_counter() + args.load_s
        i = 0
        while time.perf_counter() < t_end:
            chain.replay()
            i += 1
            if i % 8 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(chain, tails, args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    ms_max = _max_over_ranks(ms, world, dev)
    # a steadier figure beside it: the median over five more windows of the same steps
    windows = []
    for _ in range(5):
        e0.record(stream)
        run_steps(chain, tails, args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        windows.append(_max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps)
    value = whole_job_rate(B * args.steps, world, ms_max)
    ms_per_step = ms_max / args.steps
    algo_bytes_step = per_step
    hbm_gbs = algo_bytes_step / (ms_per_step / 1e3) / 1e9

    # the same steps with one graph launch per step (no overlap between steps)
    for i in range(args.warmup):
        graphs[i % n_rep].replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        graphs[i % n_rep].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_one = _max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    del graphs

    # the other variant of the step: the insert on a side stream beside the indexer (or,
    # when that is the headline, serialised before it), timed the same way
    for r in reps:
        r.side = None if side else torch.cuda.Stream(device=dev)
    alt_chain = capture(reps)
    alt_tails = {args.steps % n_rep: capture(reps[:args.steps % n_rep])} if args.steps % n_rep else {}
    for _ in range(-(-args.warmup // n_rep)):
        alt_chain.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    run_steps(alt_chain, alt_tails, args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_alt = _max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    ms_side, ms_ser = (ms_per_step, ms_alt) if side else (ms_alt, ms_per_step)
    overlap = {"ms_per_step_side_stream": ms_side, "ms_per_step_serial": ms_ser,
               "latency_saving": 1.0 - ms_side / ms_ser}
    del alt_chain, alt_tails
    for r in reps:
        r.side = torch.cuda.Stream(device=dev) if side else None

    # per-call timing over the same rotating replicas; the roofline line is the slower of
    # the two large calls (both HBM-bound by arithmetic intensity)
    calls_chained = {}
    calls = _per_call_times(reps, args.steps, stream, chained=calls_chained)
    fp4 = None if args.skip_fp4 else _fp4_indexer(w, reps, args, dev, world, hbm_peak, peak_src)
    n_vis = (L - 8) // 4 + 1
    roof = {}
    for call, kern, nbytes in (
            ("index_topk", "v4a_index_topk (indexer scores + top-k)",
             B * index_bytes_per_query(n_vis, 512)),
            ("attention", "v4a_attn_decode (attention + split merge)",
             B * attn_bytes_per_query(512, 128))):
        gbs = nbytes / (calls_chained[call] / 1e3) / 1e9
        traffic = _profile_traffic(call)
        roof[call] = {"kernel": kern, "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                      "unit": "GB/s", "frac": gbs / hbm_peak, "traffic": traffic,
                      "traffic_source": None if traffic is None else
                      "profile-sourced: dram__bytes_read.sum + dram__bytes_write.sum per call "
                      "from the committed ncu summary profiles/%s_c4a_decode_B32_L32768.md "
                      "(same library version), not measured in this run" % call,
                      "peak_source": peak_src, "algorithmic_bytes_per_launch": nbytes,
                      "us_per_launch": calls_chained[call] * 1e3,
                      "timing": "calls of consecutive replicas chained in one CUDA graph "
                                "(steady state, the way the step runs them); one graph "
                                "per call (adds the graph launch latency) beside it",
                      "us_per_launch_one_graph_per_call": calls[call] * 1e3,
                      "frac_one_graph_per_call": nbytes / (calls[call] / 1e3) / 1e9 / hbm_peak}
    dominant = max(roof, key=lambda c: calls_chained[c])
    err_bits = 0
    for r in reps:
        err_bits |= int(r.err.item())
    if fp4 is not None:
        err_bits |= fp4["device_error_bits"]

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs, random fp8 cache rows)",
        "config": {"workload": "c4a decode B=32 L=32768: insert + index/top-512 + attention",
                   "B": B, "L": L, "H": 64, "D": 512, "d_r": 64, "H_I": 64, "d_I": 128,
                   "top_k": 512, "swa": 128, "cache": "fp8 e4m3 + fp32 row scale",
                   "l2": "inputs larger than L2: %d rotating pool replicas, %.1f MB touched per "
                         "step, %.0f MB L2" % (n_rep, per_step / 1e6, l2 / 2 ** 20),
                   "launch": "one CUDA graph holds one step of each replica (%d steps, linked "
                             "by programmatic dependent launch, as a model's layers run in one "
                             "graph), replayed; %s" % (n_rep, "the insert on a side stream beside "
                             "the indexer" if side else "serial step")},
        "hbm_gbs": hbm_gbs,
        "hbm_frac": hbm_gbs / hbm_peak,
        "ms_per_step_one_graph_per_step": ms_one,
        "ms_per_step_median_of_5_windows": float(np.median(windows)),
        "ms_per_step_windows": windows,
        "per_call_ms": calls,
        "per_call_ms_chained": calls_chained,
        "side_stream": overlap,
        "fp4_indexer": fp4,
        "roofline": roof[dominant],
        "roofline_other": roof["attention" if dominant == "index_topk" else "index_topk"],
        "device_error_bits": err_bits,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if not args.skip_e2e:
        line["e2e"] = _e2e(reps, w, args.steps, dev, world)
    if not args.skip_prefill:
        line["prefill"] = _prefill(dev, tf_peak, tf_sus)
    if not args.skip_c128a:
        line["c128a_decode"] = _c128a_decode(dev, args, l2, hbm_peak, tf_peak, rank, world)
        err_bits |= line["c128a_decode"]["device_error_bits"]
    if not args.skip_mixed:
        line["mixed_decode"] = _mixed_decode(dev, args, l2, hbm_peak, rank, world)
        err_bits |= line["mixed_decode"]["device_error_bits"]
    if not args.skip_aux:
        line["compressor_aux"] = _compressor_aux(dev, hbm_peak)
        err_bits |= line["compressor_aux"]["device_error_bits"]
    line["device_error_bits"] = err_bits
    if rank == 0 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline_subprocess(2, args.cpu_budget_s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if err_bits:
        raise SystemExit("device error bits 0x%x raised during the decode steps" % err_bits)


def whole_job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processes the same units; the job takes the slowest rank's
    time, so the whole-job rate is all ranks' units over that time."""
    return world * units_per_rank / (ms_max / 1e3)


def rank_seed(rank: int) -> int:
    """Each rank's decode replica draws its own inputs (no data-path collective)."""
    return 1 + 1000 * rank


def _max_over_ranks(ms, world, dev):
    if world == 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _fp4_indexer(w8, reps8, args, dev, world, hbm_peak, peak_src):
    """The same decode step with the indexer cache in fp4 (packed e2m1 + row scale): the
    step timed like the headline (one graph holds one step of each replica) and the
    index_topk call alone, with its roofline over the fp4 bytes."""
    import torch
    import workloads as wl
    from compressed_sparse_long_gb300.layer import Layer
    w = wl.c4a_decode(seed=rank_seed(int(os.environ.get("RANK", "0"))), B=B, L=L, idx_fp4=True)
    base = Layer.from_host(w.layers[0], dev)
    n_rep = len(reps8)
    side = reps8[0].side is not None
    reps = [DecodeReplica(base, w, dev, clone=False, side=side)] + \
        [DecodeReplica(base, w, dev, clone=True, side=side) for _ in range(n_rep - 1)]
    for r in reps:
        r.step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in reps:
            r.step()
    stream = torch.cuda.current_stream()
    k = max(1, args.steps // n_rep)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(k):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_step = _max_over_ranks(e0.elapsed_time(e1), world, dev) / (k * n_rep)
    ms_idx = _per_call_times(reps, args.steps, stream, only=("index_topk",))["index_topk"]
    err = 0
    for r in reps:
        err |= int(r.err.item())
    n_vis = (L - 8) // 4 + 1
    nb = B * index_bytes_per_query(n_vis, 512, idx_fp4=True)
    gbs = nb / (ms_idx / 1e3) / 1e9
    del g
    return {"value": whole_job_rate(B * k * n_rep, world, ms_step * k * n_rep), "unit": UNIT,
            "ms_per_step": ms_step, "steps": k * n_rep, "device_error_bits": err,
            "index_topk_ms": ms_idx,
            "index_roofline": {"kernel": "v4a_index_topk over the fp4 cache", "bound": "hbm",
                               "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                               "frac": gbs / hbm_peak, "peak_source": peak_src,
                               "algorithmic_bytes_per_launch": nb},
            "bytes_per_step": reps[0].touched_bytes()}


def _per_call_times(reps, steps, stream, only=None, chained=None):
    """Device time of each library call: one CUDA graph per (call, replica), replayed
    round-robin over the replicas, timed with events on the launching stream (each replay
    pays the graph's launch latency). With `chained` (a dict), the steady-state time per
    call goes there too: one graph holds the call for every replica in turn, linked by
    programmatic dependent launch as consecutive calls run in a model, replayed."""
    import torch
    n = len(reps)
    calls = {
        "compress_insert": lambda r: r.lay.compress_insert(r.cu, r.start, r.kv, r.s, r.ik, r.is_),
        "index_topk": lambda r: r.lay.index_topk(r.q_seq, r.q_pos, r.max_pos, r.q_idx, r.w, r.topk),
        "attention": lambda r: r.lay.attention(r.q_seq, r.q_pos, r.max_pos, r.q,
                                               r.topk if r.lay.top_k else None, out=r.out),
        # the same attention with the fp8 output epilogue (e4m3 codes + per-row scales)
        "attention_q8": lambda r: r.lay.attention_q8(r.q_seq, r.q_pos, r.max_pos, r.q, r.topk),
        # the insert with the per-head query RMSNorm in the same launch, and the norm alone
        "compress_insert_qnorm": lambda r: r.lay.compress_insert_qnorm(
            r.cu, r.start, r.kv, r.s, r.ik, r.is_, r.q, r.q_gamma, q_out=r.qn),
        "q_norm_alone": lambda r: r.lay.compress_insert_qnorm(
            r.cu[:1], r.start[:0], r.kv[:0], r.s[:0], r.ik[:0], r.is_[:0], r.q, r.q_gamma,
            q_out=r.qn),
    }
    out = {}
    for name, fn in calls.items():
        if only is not None and name not in only:
            continue
        graphs = []
        for r in reps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(r)
            graphs.append(g)
        for i in range(3):
            graphs[i % n].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            graphs[i % n].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / steps
        if chained is not None:
            del graphs
            chained[name] = chained_ms_per_step([lambda r=r: fn(r) for r in reps], steps, 3,
                                                stream)
    return out


def _profile_traffic(call: str):
    """DRAM bytes per launch of a call from its committed ncu summary, if that summary still
    describes the current kernels (it states the library version)."""
    p = os.path.join(ROOT, "profiles", "%s_c4a_decode_B32_L32768.md" % call)
    if not os.path.exists(p):
        return None
    import compressed_sparse_long_gb300 as v4a
    txt = open(p).read()
    ver, traffic = None, None
    for ln in txt.splitlines():
        if ln.startswith("library_version:"):
            ver = int(ln.split(":")[1])
        if ln.startswith("traffic_bytes_per_call:"):
            traffic = float(ln.split(":")[1])
    return traffic if ver == v4a.v4a_version() else None


def _e2e(reps, w, steps, dev, world):
    """Same steps through the public API with host buffers: per step the new tokens and
    queries go host->device from a pinned buffer (one copy) and the output comes back to
    pinned memory (one copy). As on the device, one CUDA graph holds one step of every
    replica. Inputs are double-buffered the way a serving engine overlaps the next batch's
    upload with the current batch: graph X computes on device buffers X while a copy stream
    uploads the next graph's inputs into buffers Y, and each step's read-back runs on a
    second copy stream after its calls. Every step of the timed region pays one upload (the
    inputs of the same replica's next step) and one read-back; the uploads for the first
    graph happen before the timed region."""
    import torch
    b, q = w.batch, w.queries
    bf = torch.bfloat16
    fields = [(b.kv, bf), (b.s, bf), (b.ik, bf), (b.is_, bf), (q.q, bf), (q.q_idx, bf),
              (q.w, torch.float32), (b.cu, torch.int32), (b.start, torch.int64),
              (q.seq, torch.int32), (q.pos, torch.int64)]
    tensors = [torch.from_numpy(np.ascontiguousarray(x)).to(dt) for x, dt in fields]
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    n = len(reps)
    host_in, host_out = [], []
    dev_in = [[], []]       # two device input sets
    views = [[], []]
    for _ in range(n):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        for t, o in zip(tensors, offs):
            nb = t.numel() * t.element_size()
            hb[o:o + nb].copy_(t.reshape(-1).view(torch.uint8))
        host_in.append(hb)
        host_out.append(torch.empty(reps[0].out.shape, dtype=bf).pin_memory())
        for x in range(2):
            db = torch.empty(total, dtype=torch.uint8, device=dev)
            dev_in[x].append(db)
            views[x].append([db[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                             for t, o in zip(tensors, offs)])
    h2d = sum(t.numel() * t.element_size() for t in tensors)
    d2h = host_out[0].numel() * host_out[0].element_size()
    stream = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def steps_of(x, idx, up_idx):
        """Steps `idx` on input set x; uploads of `up_idx` into set 1 - x beside them."""
        main = torch.cuda.current_stream()
        up.wait_stream(main)
        down.wait_stream(main)
        with torch.cuda.stream(up):
            for i in up_idx:
                dev_in[1 - x][i].copy_(host_in[i], non_blocking=True)
        for i in idx:
            r = reps[i]
            kv, s_, ik, is_, qq, qi, ww, cu, st, qs, qp = views[x][i]
            r.lay.step(cu, st, kv, s_, ik, is_, qs, qp, r.max_pos, qq, qi, ww, out=r.out,
                       side_stream=r.side)
            e_done = torch.cuda.Event()
            e_done.record(main)
            down.wait_event(e_done)
            with torch.cuda.stream(down):
                host_out[i].copy_(r.out, non_blocking=True)
        main.wait_stream(up)
        main.wait_stream(down)

    def capture(x, idx, up_idx):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            steps_of(x, idx, up_idx)
        return g

    full = list(range(n))
    for x in range(2):                      # both input sets filled once, untimed
        for i in full:
            dev_in[x][i].copy_(host_in[i])
    steps_of(0, full, full)
    torch.cuda.synchronize()
    chains = [capture(0, full, full), capture(1, full, full)]
    n_chain, rem = steps // n, steps % n
    # the tail graph uploads the next inputs of its replicas too: every timed step pays one
    # upload and one read-back
    tail = [capture(0, range(rem), range(rem)), capture(1, range(rem), range(rem))] if rem else None
    for x in range(2):
        chains[x].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for c in range(n_chain):
        chains[c & 1].replay()
    if tail is not None:
        tail[n_chain & 1].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    # the read-back of the last graph holds each of its replicas' output
    last = range(rem) if rem else range(n)
    if not all(torch.equal(host_out[i], reps[i].out.cpu()) for i in last):
        raise SystemExit("e2e: the read-back output differs from the device output")
    ms = _max_over_ranks(e0.elapsed_time(e1), world, dev)
    uploads = n_chain * n + rem      # copies in the timed region, one per step
    return {"value": whole_job_rate(B * steps, world, ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps,
            "uploads_in_timed_region": uploads, "read_backs_in_timed_region": steps,
            "launch": "double-buffered inputs: each graph holds one step of each of the %d "
                      "replicas on one device input set while a copy stream uploads the next "
                      "graph's inputs into the other; each step's read-back on a second copy "
                      "stream" % n}


def _c128a_decode(dev, args, l2, hbm_peak, tf_peak, rank, world):
    """Dense c128a decode, B=8 sequences of 2^20 context tokens: insert + attention over
    every visible entry (8192) and the window, chained over rotating pool replicas like the
    headline; the attention call alone per replica graph; rooflines for both bounds (the
    workload sits at the ridge of HBM bandwidth and dense tensor throughput)."""
    import torch
    import workloads as wl
    from compressed_sparse_long_gb300.layer import Layer
    w = wl.c128a_decode(seed=2 + 1000 * rank)
    base = Layer.from_host(w.layers[0], dev)
    nq = len(w.queries.pos)
    L128 = int(w.queries.pos.max())
    n_vis = (L128 - 128) // 128 + 1
    per_q = c128a_bytes_per_query(n_vis, 128)
    per_step = nq * per_q["total"]
    n = n_replicas(per_step, l2, args.replicas)
    reps = [DecodeReplica(base, w, dev, clone=i > 0) for i in range(n)]
    stream = torch.cuda.current_stream()
    ms = _max_over_ranks(chained_ms_per_step([r.step for r in reps], args.steps, args.warmup,
                                             stream), world, dev)
    ch = {}
    ms_attn_one = _max_over_ranks(_per_call_times(reps, args.steps, stream, only=("attention",),
                                                  chained=ch)["attention"], world, dev)
    ms_attn = _max_over_ranks(ch["attention"], world, dev)
    attn_bytes = nq * (per_q["total"] - per_q["insert"])
    flops = nq * attn_flops_per_query(n_vis + 128)
    gbs = attn_bytes / (ms_attn / 1e3) / 1e9
    tfs = flops / (ms_attn / 1e3) / 1e12
    err = 0
    for r in reps:
        err |= int(r.err.item())
    out = {"workload": "c128a dense decode B=%d L=%d: insert + attention over %d entries + %d "
                       "window rows" % (nq, L128, n_vis, 128),
           "value": whole_job_rate(nq, world, ms), "unit": UNIT, "ms_per_step": ms,
           "bytes_per_step": per_step, "hbm_gbs": per_step / (ms / 1e3) / 1e9,
           "hbm_frac": per_step / (ms / 1e3) / 1e9 / hbm_peak, "replicas": n,
           "attention_ms": ms_attn, "attention_ms_one_graph_per_call": ms_attn_one,
           "attention_roofline": {"kernel": "v4a_attn_decode, dense (attention + split merge)",
                                  "bound": "hbm", "achieved": gbs, "peak": hbm_peak,
                                  "unit": "GB/s", "frac": gbs / hbm_peak,
                                  "algorithmic_bytes_per_launch": attn_bytes,
                                  "tensor_tflops": tfs, "tensor_frac": tfs / tf_peak,
                                  "flops_per_launch": flops},
           "device_error_bits": err}
    del reps
    return out


def _mixed_decode(dev, args, l2, hbm_peak, rank, world):
    """Mixed variable-length decode: 64 sequences with log-uniform context lengths in
    [4096, 2^20), one c4a layer (insert beside indexer + top-512, attention) and one c128a
    layer (insert, dense attention) per step; bytes exact from the drawn lengths."""
    import torch
    import workloads as wl
    from compressed_sparse_long_gb300.layer import Layer
    w = wl.mixed_decode(seed=4 + 1000 * rank)
    lens = w.meta["lens"]
    l4, l128 = (Layer.from_host(h, dev) for h in w.layers)
    nb = mixed_bytes(lens)
    n = n_replicas(nb["total"], l2, args.replicas)
    reps = [(DecodeReplica(l4, w, dev, clone=i > 0, side=True),
             DecodeReplica(l128, w, dev, clone=i > 0)) for i in range(n)]
    stream = torch.cuda.current_stream()
    both = [(lambda a=a, b=b: (a.step(), b.step())) for a, b in reps]
    ms = _max_over_ranks(chained_ms_per_step(both, args.steps, args.warmup, stream), world, dev)
    ms4 = _max_over_ranks(chained_ms_per_step([a.step for a, _ in reps], args.steps, args.warmup,
                                              stream), world, dev)
    ms128 = _max_over_ranks(chained_ms_per_step([b.step for _, b in reps], args.steps,
                                                args.warmup, stream), world, dev)
    nq = len(lens)
    err = 0
    for a, b in reps:
        err |= int(a.err.item()) | int(b.err.item())
    out = {"workload": "mixed decode B=%d, lengths log-uniform in [4096, 2^20) (min %d, max %d, "
                       "mean %.0f): one c4a layer (top-512) + one c128a layer (dense), SWA 128"
                       % (nq, min(lens), max(lens), float(np.mean(lens))),
           "value": whole_job_rate(nq, world, ms), "unit": UNIT, "ms_per_step": ms,
           "bytes_per_step": nb, "hbm_gbs": nb["total"] / (ms / 1e3) / 1e9,
           "hbm_frac": nb["total"] / (ms / 1e3) / 1e9 / hbm_peak,
           "c4a_layer": {"ms_per_step": ms4, "hbm_frac": nb["c4a_layer"] / (ms4 / 1e3) / 1e9 / hbm_peak},
           "c128a_layer": {"ms_per_step": ms128,
                           "hbm_frac": nb["c128a_layer"] / (ms128 / 1e3) / 1e9 / hbm_peak},
           "replicas": n, "device_error_bits": err}
    del reps
    return out


def _compressor_aux(dev, hbm_peak, reps=5):
    """Auxiliary compressor batch: 32 sequences of 8192 new tokens each after 4096 cached
    ones (same input distribution as the prefill chunk, seed 5), one insert call; bytes
    from the per-token count (inputs larger than L2)."""
    import torch
    import workloads as wl
    from compressed_sparse_long_gb300.layer import Layer
    spec = wl.LayerSpec("c4a", True)
    rng = np.random.default_rng(5)
    ctx, new = [4096] * 32, [8192] * 32
    bias, gamma, ibias = wl.layer_params(rng, spec)
    h = wl.make_layer(rng, spec, ctx, new, prefill_cache=True)
    h.bias, h.gamma, h.ibias = bias, gamma, ibias
    b = wl.make_batch(rng, spec, ctx, new)
    lay = Layer.from_host(h, dev)
    bf = torch.bfloat16
    cu, st = _dev(b.cu, torch.int32, dev), _dev(b.start, torch.int64, dev)
    kv, sc, ik, is_ = (_dev(x, bf, dev) for x in (b.kv, b.s, b.ik, b.is_))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        lay.compress_insert(cu, st, kv, sc, ik, is_, dev_err=err)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        lay.compress_insert(cu, st, kv, sc, ik, is_, dev_err=err)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    tokens = int(sum(new))
    nbytes = tokens * compress_bytes_per_token()
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": "auxiliary: 32 sequences x 8192 new tokens after 4096 cached (c4a, bf16 "
                        "inputs, fp8 caches)", "ms": ms, "tokens_per_s": tokens / (ms / 1e3),
            "roofline": {"kernel": "v4a_compress_insert", "bound": "hbm", "achieved": gbs,
                         "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "algorithmic_bytes_per_launch": nbytes,
                         "bytes_per_token": compress_bytes_per_token()},
            "device_error_bits": int(err.item())}


def _prefill(dev, tf_peak, tf_sus):
    """Chunked prefill: 8192 new tokens after 122880 cached; each call timed with events."""
    import torch
    import workloads as wl
    from compressed_sparse_long_gb300.layer import Layer
    w = wl.c4a_prefill(seed=3)
    lay = Layer.from_host(w.layers[0], dev)
    r = DecodeReplica(lay, w, dev, clone=False)
    r.step()
    torch.cuda.synchronize()
    reps = 3
    t = {}
    scores = None
    for name in ("compress_insert", "index_topk", "index_scores", "attention"):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            if name == "compress_insert":
                r.lay.compress_insert(r.cu, r.start, r.kv, r.s, r.ik, r.is_)
            elif name == "index_topk":
                r.lay.index_topk(r.q_seq, r.q_pos, r.max_pos, r.q_idx, r.w, r.topk)
            elif name == "index_scores":
                scores = r.lay.index_scores(r.q_seq, r.q_pos, r.max_pos, r.q_idx, r.w)
            else:
                r.lay.attention(r.q_seq, r.q_pos, r.max_pos, r.q, r.topk, out=r.out,
                                prefill=True)
        e1.record()
        torch.cuda.synchronize()
        t[name] = e0.elapsed_time(e1) / reps
    del scores
    t["topk"] = t["index_topk"] - t["index_scores"]
    n_q = len(w.queries.pos)
    flops = n_q * attn_flops_per_query(512 + 128)
    pos = w.queries.pos
    idx_flops = float(sum(((p - 8) // 4 + 1) for p in pos)) * 2 * 64 * 128
    step = t["compress_insert"] + t["index_topk"] + t["attention"]
    cbytes = n_q * compress_bytes_per_token()
    cgbs = cbytes / (t["compress_insert"] / 1e3) / 1e9
    return {"workload": "c4a prefill: 122880 cached + 8192-token chunk",
            "attn_tflops": flops / (t["attention"] / 1e3) / 1e12,
            "attn_frac_of_bf16_peak": flops / (t["attention"] / 1e3) / 1e12 / tf_peak,
            "indexer_tflops": idx_flops / (t["index_topk"] / 1e3) / 1e12,
            "indexer_scores_tflops": idx_flops / (t["index_scores"] / 1e3) / 1e12,
            "indexer_scores_frac_of_bf16_peak": idx_flops / (t["index_scores"] / 1e3) / 1e12 / tf_peak,
            "tokens_per_s": n_q / (step / 1e3), "ms": t,
            "ms_note": "topk = index_topk - index_scores (the call's selection kernel)",
            "compress_tokens_per_s": n_q / (t["compress_insert"] / 1e3),
            "compress_roofline": {"kernel": "v4a_compress_insert (8192-token chunk)",
                                  "bound": "hbm", "achieved": cgbs, "peak": hbm_peak_of(),
                                  "unit": "GB/s", "frac": cgbs / hbm_peak_of(),
                                  "algorithmic_bytes_per_launch": cbytes,
                                  "bytes_per_token": compress_bytes_per_token()}}


def hbm_peak_of() -> float:
    return peaks()[0]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--load-s", type=float, default=1.5, dest="load_s")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0, dest="cpu_budget_s")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-fp4", action="store_true", dest="skip_fp4")
    ap.add_argument("--serial-step", action="store_true", dest="serial_step",
                    help="time the serial step as the headline (default: the decode insert on a "
                         "side stream beside the indexer; the other variant is reported beside it)")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--replicas", type=int, default=0, help="pool replicas (0: enough to exceed 4x L2)")
    ap.add_argument("--skip-c128a", action="store_true", dest="skip_c128a")
    ap.add_argument("--skip-mixed", action="store_true", dest="skip_mixed")
    ap.add_argument("--skip-aux", action="store_true", dest="skip_aux")
    ap.add_argument("--only", choices=["all", "prefill", "c128a", "mixed", "compress"],
                    default="all")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_main(args, rank)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    gpu_main(args, rank, world, local_rank)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
