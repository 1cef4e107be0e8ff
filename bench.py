"""Benchmark of one DSA layer step (indexer -> top-k -> slots -> sparse MLA).

Default workload: decode at 128K context, batch 8, FP8 latents (576 B) and
FP8 index keys (132 B), 96 MLA heads, 32 indexer heads, top-k 2048, page 64.
Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

value      query-tokens/s of the whole job (inputs resident in HBM), timed over CUDA
           graphs of consecutive steps that carry no event nodes: the median of 5 timed
           regions of exactly K steps each (all five in `repeats_ms_per_step`)
clocks     nvidia-smi samples over the timed regions and 0.6 s more of the same steps
e2e        the same through the C ABI with host buffers: pinned host -> device
           copies of the step's queries and metadata and device -> host copies of
           the outputs inside the timed region, one graph replay per step between them
roofline   the indexer (the dominant kernel): algorithmic bytes per launch /
           its launch duration (the step's scorer calls launched back to back in one
           CUDA graph over the same rotating cache copies, events at the graph's two
           ends), against the measured HBM copy bandwidth;
           prefill: FLOP per launch against the FP8 GEMM peak measured in the run
cpu_baseline  the CPU oracle on a bounded sample of the same workload
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "DSA decode query-tokens/s per layer at 128K ctx; achieved HBM GB/s vs ~8 TB/s"
UNIT = "query-tokens/s"
FALLBACK_HBM_GBS = 6800.0
ROTATE = 4  # independent copies of the caches; a step never re-reads what the last 3 steps read


FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 vs 2.25 PFLOP/s)


def _peaks():
    """(HBM GB/s, dense FP8 TFLOP/s, source): measured copy bandwidth and cuBLAS bf16 burst
    throughput of the GB300s; FP8 = measured bf16 x the nominal FP8/bf16 ratio."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d.get("hbm_gbs", FALLBACK_HBM_GBS)),
                float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) * FP8_OVER_BF16, "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS * FP8_OVER_BF16, "fallback"


def max_over_ranks(v: float, dist) -> float:
    """The largest of every rank's value (the slowest rank's time); `dist` None = one process."""
    if dist is None:
        return float(v)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, rows: int, steps: int, ms: float) -> float:
    """Whole-job query-tokens/s of `world` replicas that each ran `steps` steps of `rows` query
    rows in `ms` (the slowest rank's) milliseconds."""
    return world * rows * steps / (ms / 1000.0)


def indexer_flops(wl) -> int:
    """2 * 32 heads * 128 dims per (query row, visible key) pair."""
    return int(2 * 32 * 128 * int(wl.row_ctx().astype(np.int64).sum()))


class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock and throttle reasons, each stamped with
    the host time it arrived; `summary(t0, t1)` keeps those taken during [t0, t1]."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, timeout=5.0):
        t_end = time.time() + timeout
        while self.proc is not None and not self.lines and time.time() < t_end:
            time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [(t, ln) for t, ln in self.lines if t0 <= t <= t1 + 0.05]
        for _, ln in window:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


REPEATS = 5  # timed regions of K steps each; the line reports their median


def dsa_config(wl, copies: int, cache_bytes: int, world: int, single_pass: bool) -> dict:
    """The `config` object of a DSA line (the GPU arm and the reference arm print the same one)."""
    from prefill_dsa_indexer_gb300 import inputs as I
    return {"workload": wl.name, "batch": len(wl.ctx), "rows": wl.num_rows, "ctx": wl.ctx[0], "k": wl.k,
            "heads": wl.heads, "index_heads": 32, "page": 64, "key_bytes": I.INDEX_TOKEN_BYTES[wl.key_fmt],
            "latent_bytes": I.LATENT_TOKEN_BYTES[wl.lat_fmt],
            "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
            "topk": "single pass (scorer histogram)" if single_pass else "cluster radix select",
            "l2": f"inputs > L2: {copies} rotating copies of the caches ({cache_bytes * copies / 1e9:.2f} GB)"}


def measure_fp8_peak(n: int = 8192, reps: int = 10, sustain_s: float = 1.0) -> dict:
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of this GPU through the library (torch._scaled_mm,
    cuBLASLt), n^3: the best of `reps` timed calls (burst) and the mean over back-to-back calls for
    about `sustain_s` seconds (sustained), in TFLOP/s (2 n^3 per call)."""
    a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()  # column-major operand
    one = torch.ones((), device="cuda", dtype=torch.float32)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16, use_fast_accum=True)

    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    flop = 2.0 * n ** 3
    calls, t0 = 0, time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    while time.perf_counter() - t0 < sustain_s:
        for _ in range(20):
            mm()
        calls += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    return {"burst_tflops": flop / (best / 1e3) / 1e12, "sustained_tflops": flop * calls / (e0.elapsed_time(e1) / 1e3) / 1e12,
            "how": f"torch._scaled_mm e4m3 x e4m3 -> bf16, {n}^3, best of {reps} (burst), {calls} back-to-back "
                   f"calls (sustained)"}


def oracle_single_thread_ms(workload: str = "decode_tiny_4k") -> dict:
    """One whole step of the smallest workload (indexer, top-k, slots, attention) on one host thread."""
    import oracle
    from prefill_dsa_indexer_gb300 import inputs as I
    wl = I.workload(workload)
    inp = I.make_inputs(wl, device="cpu")
    h = {n: inp.np(n) for n in ("idx_pool", "lat_pool", "block_table", "row_req", "row_ctx", "q_idx", "head_w", "q_mla")}
    lib = oracle.load()
    before = lib.oracle_num_threads()
    lib.oracle_set_num_threads(1)
    try:
        t0 = time.perf_counter()
        lg = oracle.indexer_logits(h["idx_pool"], wl.key_fmt, h["block_table"], h["row_req"], h["row_ctx"], h["q_idx"],
                                   h["head_w"])
        idx = oracle.topk_f64(lg, h["row_ctx"], wl.k)
        sl = oracle.page_to_slot(h["block_table"], h["row_req"], idx)
        oracle.sparse_mla(h["lat_pool"], wl.lat_fmt, inp.tensor_scale, h["q_mla"], sl, 1.0 / np.sqrt(192.0))
        ms = (time.perf_counter() - t0) * 1e3
    finally:
        lib.oracle_set_num_threads(before)
    return {"workload": workload, "ms_per_step": ms, "threads": 1}


def indexer_algorithmic_bytes(wl, token_bytes: int) -> int:
    """Bytes the indexer must move per launch: every cached key of every row group once
    (132 B/token FP8), the block-table entries, the queries and head weights, and the
    fp32 logits it writes."""
    R = wl.num_rows
    rc = wl.row_ctx()
    groups = R // wl.rows_per_group
    gmax = [int(rc[g * wl.rows_per_group:(g + 1) * wl.rows_per_group].max()) for g in range(groups)]
    keys = sum(token_bytes * L + 4 * ((L + 63) // 64) for L in gmax)
    return keys + R * (32 * 128 + 32 * 4) + 4 * int(rc.sum())


def layer_algorithmic_bytes(wl, idx_bytes: int, lat_bytes: int) -> int:
    """The method's own traffic for one layer step: index keys once per row group, the
    selected latents (min(L, k) per row; union over a group's rows is approximated by the
    largest row), queries, outputs and block-table entries.  Logits and indices are
    implementation overhead and are not counted."""
    rc = wl.row_ctx()
    G = wl.rows_per_group
    tot = 0
    for g in range(wl.num_rows // G):
        Lg = int(rc[g * G:(g + 1) * G].max())
        tot += idx_bytes * Lg + 4 * ((Lg + 63) // 64) + lat_bytes * min(Lg, wl.k)
    R = wl.num_rows
    tot += R * (32 * 128 + 32 * 4)          # indexer query + head weights
    tot += R * wl.heads * 576 * 2           # MLA query (bf16)
    tot += R * wl.heads * (512 + 1) * 4     # output + lse (fp32)
    return tot


def run_reference(args, wl, rank):
    """The CPU oracle, as it stands, on a bounded sample per step of the same workload.

    Each step takes one whole query row (indexer scan over all its cached keys, top-k, slots,
    sparse MLA of all heads) on every host thread.  Only when a whole row would not fit the
    time budget (K + W steps in about two and a half minutes) does a step take the indexer
    over the first S keys and the MLA of H_s heads, the row's cost then extrapolated linearly
    in keys and heads (said in the line's `sample`)."""
    import oracle
    from prefill_dsa_indexer_gb300 import inputs as I
    inp = I.make_inputs(wl, device="cuda" if torch.cuda.is_available() else "cpu")
    host = {n: inp.np(n) for n in ("idx_pool", "lat_pool", "block_table", "row_req", "row_ctx", "q_idx", "head_w",
                                    "q_mla")}
    L = int(host["row_ctx"][0])
    H = wl.heads
    sm = 1.0 / np.sqrt(192.0)
    cores = oracle.num_threads()  # the row's indexer chunks and attention heads run on every thread

    def part(S, Hs, r=0):
        rr = np.array([r])
        ctx = np.array([S], dtype=np.int32)
        t0 = time.perf_counter()
        lg = oracle.indexer_logits(host["idx_pool"], wl.key_fmt, host["block_table"], host["row_req"][rr], ctx,
                                   host["q_idx"][rr], host["head_w"][rr])
        idx = oracle.topk_f64(lg, ctx, wl.k)
        sl = oracle.page_to_slot(host["block_table"], host["row_req"][rr], idx)
        t1 = time.perf_counter()
        oracle.sparse_mla(host["lat_pool"], wl.lat_fmt, inp.tensor_scale,
                          np.ascontiguousarray(host["q_mla"][rr, :Hs]), sl, sm)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    budget = max(0.01, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    ti, tm = part(L, H)
    if ti + tm <= budget:  # whole rows fit the budget: nothing is extrapolated
        S, Hs = L, H
    else:
        S = int(min(L, max(wl.k, (0.5 * budget / max(ti, 1e-6)) * L)))
        Hs = int(max(1, min(H, (0.5 * budget / max(tm, 1e-6)) * H)))
    for _ in range(args.warmup):
        part(S, Hs)
    est, wall = 0.0, 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        a, b = part(S, Hs, i % wl.num_rows)
        est += a * L / S + b * H / Hs
    wall = time.perf_counter() - t0
    value = args.steps / est
    sample = (f"per step 1 of {wl.num_rows} query rows of {wl.name}: indexer + top-k over {S} of its {L} keys, "
              f"sparse MLA of {Hs} of {H} heads over the selected tokens"
              + ("" if (S, Hs) == (L, H) else "; full-row time extrapolated linearly (keys, heads)")
              + f"; {cores} threads, {wall:.1f} s of CPU work")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * est / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dsa_config(wl, max(1, args.copies), inp.idx_pool.numel() + inp.lat_pool.numel(), args.gpus,
                                 args.single_pass),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if rank == 0:
        print(json.dumps(line), flush=True)


def cpu_baseline(wl, inp, budget_s=12.0):
    """The oracle on whole rows of the workload, cycling over the rows until about budget_s of wall
    time, on every host thread (OpenMP over (row, token chunk) for the indexer, (row, head) for the
    attention)."""
    import oracle
    host = {n: inp.np(n) for n in ("idx_pool", "lat_pool", "block_table", "row_req", "row_ctx", "q_idx", "head_w",
                                    "q_mla")}
    threads = oracle.num_threads()
    done, t_used, n = 0, 0.0, 1
    while t_used < budget_s:
        rows = (np.arange(n) + done) % wl.num_rows
        t0 = time.perf_counter()
        lg = oracle.indexer_logits(host["idx_pool"], wl.key_fmt, host["block_table"], host["row_req"][rows],
                                   host["row_ctx"][rows], host["q_idx"][rows], host["head_w"][rows])
        idx = oracle.topk_f64(lg, host["row_ctx"][rows], wl.k)
        sl = oracle.page_to_slot(host["block_table"], host["row_req"][rows], idx)
        oracle.sparse_mla(host["lat_pool"], wl.lat_fmt, inp.tensor_scale, host["q_mla"][rows], sl,
                          1.0 / np.sqrt(192.0))
        t_used += time.perf_counter() - t0
        done += len(rows)
    return {"value": done / t_used, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{done} query rows of {wl.name} (whole rows: full indexer scan, top-k, MLA), one row "
                      f"per call on {threads} threads, {t_used:.1f} s",
            "single_thread": oracle_single_thread_ms()}


def msa_score_bytes(wl) -> int:
    """Bytes the MSA block-score scan must move per launch: every visible index key of every
    row group once (128 B/token), the block-table entries, the index queries and the fp32
    block scores it writes."""
    rc = wl.row_ctx()
    G = wl.rows_per_group
    tot = 0
    for g in range(wl.num_rows // G):
        Lg = int(rc[g * G:(g + 1) * G].max())
        tot += 128 * Lg + 4 * ((Lg + 127) // 128)
    return tot + wl.num_rows * 4 * 128 + 4 * 4 * int(((rc + 127) // 128).sum())


def msa_layer_bytes(wl) -> int:
    """The MSA step's own traffic: index keys once per row group, each (row, group)'s
    selected K and V (min(L, 2048) tokens x 256 B), queries, outputs and lse."""
    rc = wl.row_ctx()
    H = 4 * wl.heads_per_group
    tot = msa_score_bytes(wl)
    tot += sum(4 * 256 * min(int(L), 2048) for L in rc)
    tot += wl.num_rows * H * 128                # FP8 attention queries
    tot += wl.num_rows * H * (128 + 1) * 4      # output + lse (fp32)
    return tot


def run_msa(args, rank, world, local, dist):
    """One MSA block-sparse step (block scores -> selection -> attention) per query row batch."""
    from prefill_dsa_indexer_gb300 import inputs as I
    wl = I.msa_workload(args.workload)
    metric = "MSA decode query-tokens/s per layer; achieved HBM GB/s of the block-score scan"
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import prefill_dsa_indexer_gb300 as P
    inp = I.make_msa_inputs(wl, device="cuda")
    R, H = wl.num_rows, 4 * wl.heads_per_group
    sm = 1.0 / np.sqrt(128.0)
    copies = max(1, args.copies)
    pools = [(inp.idx_pool, inp.kv_pool)] + [(inp.idx_pool.clone(), inp.kv_pool.clone()) for _ in range(copies - 1)]
    nb = (inp.max_ctx + 127) // 128
    scores = torch.empty((R, 4, nb), dtype=torch.float32, device="cuda")
    blocks = torch.empty((R, 4, 16), dtype=torch.int32, device="cuda")
    out = torch.empty((R, H, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((R, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(P.msa_attention_workspace_size(R, wl.heads_per_group), dtype=torch.uint8, device="cuda")
    st = P.new_status()

    def step(i, q=inp.q, q_idx=inp.q_idx, ev=None, s=None):
        ip, kp = pools[i % len(pools)]
        if ev is not None:
            ev[0].record(s)
        P.msa_block_scores(ip, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, q_idx, wl.rows_per_group,
                           scores=scores, status=st, stream=s)
        if ev is not None:
            ev[1].record(s)
        P.msa_select(scores, inp.row_ctx, inp.max_ctx, blocks=blocks, status=st, stream=s)
        P.msa_attention(kp, inp.k_scale, inp.v_scale, inp.block_table, inp.row_req, inp.row_ctx, inp.max_ctx, q,
                        inp.q_scale, blocks, sm, out=out, lse=lse, workspace=ws, status=st, stream=s)

    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        step(i, s=stream)
    torch.cuda.synchronize()
    P.check_status(st, "warm-up")
    # CUDA graphs of 16 x copies consecutive steps; a second graph of the same steps carries event
    # nodes around every block-score launch and is replayed after the timed loop to time them
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    n = 16 * copies
    g, gp = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    evp = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
           for _ in range(n)]
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for k in range(n):
                step(k, s=cap)
        with torch.cuda.graph(gp, stream=cap):
            for k in range(n):
                step(k, ev=evp[k], s=cap)
    stream.wait_stream(cap)
    g.replay()
    gp.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // n)
    steps = reps * n
    rep_ms = []
    with ClockSampler(local) as clk:  # REPEATS timed regions, then >= 0.6 s more of the same steps
        clk.wait_first()
        h0 = time.time()
        for _rep in range(REPEATS):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if dist is not None:
                dist.barrier()
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            t1.record(stream)
            torch.cuda.synchronize()
            if dist is not None:
                dist.barrier()
            rep_ms.append(t0.elapsed_time(t1))
        h1 = time.time()
        while time.time() - h1 < 0.6:
            g.replay()
            torch.cuda.synchronize()
        h2 = time.time()
    total_ms = statistics.median(rep_ms)
    total_ms = max_over_ranks(total_ms, dist)
    P.check_status(st, "timed steps")
    for _ in range(3):
        gp.replay()
    torch.cuda.synchronize()
    score_ms = sum(a.elapsed_time(b) for a, b in evp) / len(evp)
    value = replica_throughput(world, R, steps, total_ms)
    # end to end: queries in from pinned host memory, outputs back, inside the timed region
    hq, hqi = inp.q.cpu().pin_memory(), inp.q_idx.cpu().pin_memory()
    dq, dqi = torch.empty_like(inp.q), torch.empty_like(inp.q_idx)
    ho, hl = torch.empty(out.shape, dtype=torch.float32).pin_memory(), torch.empty(lse.shape).pin_memory()
    # one CUDA graph per cache copy for the step between the copies
    ge = [torch.cuda.CUDAGraph() for _ in range(copies)]
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for c in range(copies):
            with torch.cuda.graph(ge[c], stream=cap):
                step(c, q=dq, q_idx=dqi, s=cap)
    stream.wait_stream(cap)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            e0.record(stream)
        dq.copy_(hq, non_blocking=True)
        dqi.copy_(hqi, non_blocking=True)
        with torch.cuda.stream(stream):
            ge[i % copies].replay()
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    P.check_status(st, "e2e steps")
    e2e_ms = e0.elapsed_time(e1)
    hbm_peak, _, peak_kind = _peaks()
    sb = msa_score_bytes(wl)
    achieved = sb / (score_ms / 1000.0) / 1e9
    lb = msa_layer_bytes(wl)
    msa_traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            msa_traffic = json.load(f).get(wl.name)
    line = {
        "metric": metric, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": total_ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3xe4m3->f32 (scores, S), f16xf16->f32 (PV)", "data": "synthetic",
        "config": {"workload": wl.name, "batch": len(wl.ctx), "rows": R, "ctx": wl.ctx[0], "groups": 4,
                   "heads_per_group": wl.heads_per_group, "blocks": 16, "page": 128,
                   "l2": f"inputs > L2: {copies} rotating copies of the caches "
                         f"({(inp.idx_pool.numel() + inp.kv_pool.numel()) * copies / 1e9:.2f} GB)"},
        "layer_hbm_gbs": lb / (total_ms / steps / 1000.0) / 1e9, "layer_algorithmic_bytes": lb,
        "roofline": {"kernel": f"msa_scores_kernel<{wl.rows_per_group}>", "bound": "hbm", "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                     "algorithmic_bytes": sb, "ms_per_launch": score_ms, "traffic": msa_traffic},
        "e2e": {"value": replica_throughput(world, R, args.steps, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": hq.numel() + hqi.numel(), "d2h_bytes_per_step": (ho.numel() + hl.numel()) * 4,
                "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": 4 * steps,
        "launch": f"CUDA graphs of {n} consecutive steps; block scores timed after the timed loop by event "
                  f"nodes around each launch in a replay of the same steps",
        "repeats_ms_per_step": [m / steps for m in rep_ms],
        "clocks": dict(clk.summary(h0, h2), window=f"the {REPEATS} timed regions and {h2 - h1:.2f} s of the "
                                                       f"same steps right after them"),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        host = {k: inp.np(k) for k in ("idx_pool", "kv_pool", "block_table", "row_req", "row_ctx", "q_idx", "q")}
        done, used = 0, 0.0
        while used < 12.0:
            rows = np.array([done % R])
            ta = time.perf_counter()
            sc = oracle.msa_block_scores(host["idx_pool"], host["block_table"], host["row_req"][rows],
                                         host["row_ctx"][rows], host["q_idx"][rows])
            bl = oracle.msa_select(sc, host["row_ctx"][rows])
            oracle.msa_attention(host["kv_pool"], inp.k_scale, inp.v_scale, host["block_table"],
                                 host["row_req"][rows], host["row_ctx"][rows], host["q"][rows], inp.q_scale, bl, sm)
            used += time.perf_counter() - ta
            done += 1
        line["cpu_baseline"] = {"value": done / used, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{done} whole query rows of {wl.name} (block scores over every key, "
                                          f"selection, attention of all heads), one row per call, {used:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--copies", type=int, default=ROTATE, help="independent cache copies rotated across steps")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_b8_128k_fp8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch kernels one by one instead of graph replays")
    ap.add_argument("--single-pass", action="store_true",
                    help="scorer builds each row's logit histogram and the top-k starts from it")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    if args.workload.startswith("msa_") and args.impl == "ours":
        run_msa(args, rank, world, local, dist)
        if dist is not None:
            dist.destroy_process_group()
        return

    from prefill_dsa_indexer_gb300 import inputs as I
    wl = I.workload(args.workload)

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import prefill_dsa_indexer_gb300 as P

    inp = I.make_inputs(wl, device="cuda")
    prefill = wl.rows_per_req > 8
    layers = []
    copies = max(1, args.copies)
    for c in range(copies):
        idx_pool = inp.idx_pool if c == 0 else inp.idx_pool.clone()
        lat_pool = inp.lat_pool if c == 0 else inp.lat_pool.clone()
        layers.append(P.Layer(idx_pool, wl.key_fmt, lat_pool, wl.lat_fmt, inp.tensor_scale, inp.block_table,
                              inp.max_ctx, wl.num_rows, wl.heads, wl.k, wl.rows_per_group, prefill=prefill,
                              single_pass=args.single_pass))
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        L = layers[i % len(layers)]
        if ev is not None:
            ev[0].record(stream)
        L.score(inp.row_req, inp.row_ctx, inp.q_idx, inp.head_w, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        L.select(inp.row_req, inp.row_ctx, inp.q_mla, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    for L in layers:
        P.check_status(L.status, "warm-up")

    # Runs of consecutive steps (cycling the cache copies, as a captured multi-layer forward
    # would) are captured as one CUDA graph each, with event-record nodes around every indexer
    # launch: the indexer's time is then read on the device, free of host and graph-launch
    # latency.  Without event-record nodes (older torch) each step is two graphs with stream
    # events between them.
    def ext_event():
        return torch.cuda.Event(enable_timing=True, external=True)

    def rest_of_step(L, s=None):  # top-k (from the scorer's histogram), page -> slot, sparse MLA
        L.select(inp.row_req, inp.row_ctx, inp.q_mla, stream=s)

    def indexer(L, s=None):  # scorer: logits and their per-row histogram
        L.score(inp.row_req, inp.row_ctx, inp.q_idx, inp.head_w, stream=s)

    graph_mode = "eager"
    runs = []  # (graph, [(event before, event after) per step])
    if not args.no_graph:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        per_graph = 16 * len(layers)
        try:
            ext_event()
            graph_mode = "multi-step"
        except TypeError:
            graph_mode = "two-graphs"

        side = torch.cuda.Stream()

        def capture(n, events):
            # per step: scorer -> top-k+slots -> attention on the main branch; the decode query
            # prep (it needs only the query) forks onto a side branch after the scorer, runs beside
            # the top-k (which occupies few SMs) and joins before the attention.
            # events: event nodes around every scorer launch (the indexer timing graph only)
            g = torch.cuda.CUDAGraph()
            evp = [(ext_event(), ext_event()) for _ in range(n)] if events else []
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    for k in range(n):
                        L = layers[k % len(layers)]
                        fork = not L.prefill
                        if events:
                            evp[k][0].record(cap)
                        indexer(L)
                        if events:
                            evp[k][1].record(cap)
                        if fork:
                            side.wait_stream(cap)
                            with torch.cuda.stream(side):
                                L.prepare(inp.q_mla)
                        L.select_tokens(inp.row_req, inp.row_ctx)
                        if fork:
                            cap.wait_stream(side)
                        L.attend(inp.q_mla, prepared=fork)
            return g, evp

        if graph_mode == "multi-step":
            full, tail = divmod(args.steps, per_graph)
            if full:
                runs.append((capture(per_graph, False), full))
            if tail:
                runs.append((capture(tail, False), 1))
            # the indexer's launches are timed in a separate replay of the same steps with event
            # nodes around each scorer launch, after the timed loop
            probe = capture(min(per_graph, args.steps), True)
        else:
            pairs = []
            for c in range(len(layers)):
                g_idx, g_rest = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.stream(cap):
                    with torch.cuda.graph(g_idx, stream=cap):
                        indexer(layers[c])
                    with torch.cuda.graph(g_rest, stream=cap):
                        rest_of_step(layers[c])
                pairs.append((g_idx, g_rest))
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        for (g, _), _n in runs:  # graph warm-up: one replay of each run
            g.replay()
        if graph_mode == "multi-step":
            probe[0].replay()
        if graph_mode == "two-graphs":
            for i in range(args.warmup):
                g_idx, g_rest = pairs[i % len(pairs)]
                g_idx.replay()
                g_rest.replay()
        torch.cuda.synchronize()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def timed_steps():  # exactly args.steps steps
        if graph_mode == "multi-step":
            for (g, _), reps in runs:
                for _r in range(reps):
                    g.replay()
        elif graph_mode == "two-graphs":
            for i in range(args.steps):
                g_idx, g_rest = pairs[i % len(pairs)]
                evs[i][0].record(stream)
                g_idx.replay()
                evs[i][1].record(stream)
                g_rest.replay()
        else:
            for i in range(args.steps):
                step(i, evs[i])

    # REPEATS timed regions of exactly args.steps steps, each bracketed by a barrier and a device
    # synchronisation; the line reports their median.  nvidia-smi samples the clocks throughout and
    # over a further >= 0.6 s of the same steps right after, so short timed regions still come with
    # clock samples under the same load.
    rep_ms = []
    with ClockSampler(local) as clk:
        clk.wait_first()
        h0 = time.time()
        for _rep in range(REPEATS):
            t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            if dist is not None:
                dist.barrier()
            torch.cuda.synchronize()
            t_start.record(stream)
            timed_steps()
            t_stop.record(stream)
            torch.cuda.synchronize()
            if dist is not None:
                dist.barrier()
            rep_ms.append(t_start.elapsed_time(t_stop))
        h1 = time.time()
        while time.time() - h1 < 0.6:
            timed_steps()
            torch.cuda.synchronize()
        h2 = time.time()
    total_ms = statistics.median(rep_ms)
    if graph_mode == "multi-step":
        for _r in range(3):
            probe[0].replay()
        torch.cuda.synchronize()
        samples = [a.elapsed_time(b) for a, b in probe[1]]  # every step of the last replay
    else:
        samples = [a.elapsed_time(b) for a, b in evs]
    idx_ms_events = sum(samples) / len(samples)
    # The indexer's launch duration for the roofline: back-to-back launches of the timed steps'
    # scorer calls (same layers and cache copies, inputs > L2) in one CUDA graph, timed by events at
    # its two ends only.  An event node around every launch (idx_ms_events, also reported) adds some
    # microseconds per launch.
    idx_ms = idx_ms_events
    if graph_mode == "multi-step":
        n_idx = 16 * len(layers)
        g_idx = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g_idx, stream=cap):
                for j in range(n_idx):
                    indexer(layers[j % len(layers)])
        stream.wait_stream(cap)
        g_idx.replay()
        torch.cuda.synchronize()
        reps = []
        for _r in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_idx.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            reps.append(e0.elapsed_time(e1) / n_idx)
        idx_ms = statistics.median(reps)
    for L in layers:
        P.check_status(L.status, "timed steps")
    total_ms = max_over_ranks(total_ms, dist)
    ms_per_step = total_ms / args.steps
    value = replica_throughput(world, wl.num_rows, args.steps, total_ms)

    # ---- end to end through the C ABI with host buffers.  Every step copies its inputs from
    # pinned host memory and its outputs back; the copies run on their own streams, double
    # buffered, so step i + 1's inputs travel while step i computes and step i's outputs
    # travel while step i + 1 computes (the timed region still holds every copy).
    # A step's inputs sit in one pinned host block (each at a 256-byte aligned offset) and move
    # with one copy; the results (outputs and lse, one device buffer per layer) with one more.
    names = ("row_req", "row_ctx", "q_idx", "head_w", "q_mla")
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += (getattr(inp, n).numel() * getattr(inp, n).element_size() + 255) // 256 * 256
    pinned = torch.empty(total, dtype=torch.uint8).pin_memory()
    for n in names:
        t = getattr(inp, n).contiguous()
        nb = t.numel() * t.element_size()
        pinned[offs[n]:offs[n] + nb].copy_(t.cpu().view(-1).view(torch.uint8))
    dev_blk = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]

    def view_of(blk, n):
        t = getattr(inp, n)
        nb = t.numel() * t.element_size()
        return blk[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)

    dev_in = [{n: view_of(dev_blk[b], n) for n in names} for b in range(2)]
    host_res = [torch.empty(layers[0].outputs.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(getattr(inp, n).numel() * getattr(inp, n).element_size() for n in names)
    d2h = host_res[0].numel() * 4
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_issue(n_steps, main, body):
        # n_steps steps: step i's inputs copy in on h2d_s while step i - 1 computes on `main`, and
        # its results copy out on d2h_s while step i + 1 computes; events carry the buffer reuse
        in_ready = [torch.cuda.Event() for _ in range(n_steps)]
        done = [torch.cuda.Event() for _ in range(n_steps)]
        out_copied = [torch.cuda.Event() for _ in range(n_steps)]
        h2d_s.wait_stream(main)
        d2h_s.wait_stream(main)

        def h2d_copy(i):
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(done[i - 2])  # step i - 2 has read this input buffer
                dev_blk[i % 2].copy_(pinned, non_blocking=True)
                in_ready[i].record(h2d_s)

        h2d_copy(0)
        for i in range(n_steps):
            if i + 1 < n_steps:
                h2d_copy(i + 1)
            L = layers[i % len(layers)]
            main.wait_event(in_ready[i])
            if i >= len(layers):
                main.wait_event(out_copied[i - len(layers)])  # this layer's outputs were copied out
            with torch.cuda.stream(main):
                body(i, L, dev_in[i % 2])
            done[i].record(main)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[i])
                if i >= 2:
                    d2h_s.wait_event(out_copied[i - 2])  # host buffer i % 2 is free again
                host_res[i % 2].copy_(L.outputs, non_blocking=True)
                out_copied[i].record(d2h_s)
        main.wait_stream(d2h_s)
        main.wait_stream(h2d_s)

    def eager_body(i, L, d):
        L.run(d["row_req"], d["row_ctx"], d["q_idx"], d["head_w"], d["q_mla"], stream=torch.cuda.current_stream())

    side_e = torch.cuda.Stream()

    def graph_body(i, L, d):  # the query prep forks onto a parallel branch beside the top-k
        cur = torch.cuda.current_stream()
        fork = not L.prefill
        L.score(d["row_req"], d["row_ctx"], d["q_idx"], d["head_w"])
        if fork:
            side_e.wait_stream(cur)
            with torch.cuda.stream(side_e):
                L.prepare(d["q_mla"])
        L.select_tokens(d["row_req"], d["row_ctx"])
        if fork:
            cur.wait_stream(side_e)
        L.attend(d["q_mla"], prepared=fork)

    # With graphs, each step between its copies is one replay of a graph of that step's calls,
    # one graph per input buffer and cache copy.  (Capturing the copies too, as memcpy nodes in
    # graphs of many steps, was no faster for decode and slower for the prefill's large copies.)
    e2e_graphs = None
    if graph_mode != "eager":
        cap_e = torch.cuda.Stream()
        cap_e.wait_stream(stream)
        e2e_graphs = []
        for b in range(2):
            row = []
            for L in layers:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(cap_e):
                    with torch.cuda.graph(g, stream=cap_e):
                        graph_body(0, L, dev_in[b])
                row.append(g)
            e2e_graphs.append(row)
        stream.wait_stream(cap_e)
        torch.cuda.synchronize()

    def replay_body(i, L, d):
        e2e_graphs[i % 2][i % len(layers)].replay()

    body = replay_body if e2e_graphs is not None else eager_body
    e2e_issue(args.warmup, stream, body)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_issue(args.steps, stream, body)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dist)
    for L in layers:
        P.check_status(L.status, "e2e steps")
    e2e_value = replica_throughput(world, wl.num_rows, args.steps, e2e_ms)

    idx_tok = I.INDEX_TOKEN_BYTES[wl.key_fmt]
    lat_tok = I.LATENT_TOKEN_BYTES[wl.lat_fmt]
    idx_bytes = indexer_algorithmic_bytes(wl, idx_tok)
    layer_bytes = layer_algorithmic_bytes(wl, idx_tok, lat_tok)
    hbm_peak, fp8_peak, peak_kind = _peaks()
    if prefill:
        flops = indexer_flops(wl)
        achieved = flops / (idx_ms / 1000.0) / 1e12
        fp8 = measure_fp8_peak()
        roof = {"kernel": "indexer_kernel<8, fp8 keys>", "bound": "tensor", "achieved": achieved,
                "timing": "back-to-back launches of the step's scorer calls in one CUDA graph, events at its ends",
                "ms_per_launch_event_nodes": idx_ms_events,
                "peak": fp8["burst_tflops"], "unit": "TFLOP/s", "frac": achieved / fp8["burst_tflops"],
                "peak_kind": f"measured in this run: {fp8['how']}",
                "frac_of_sustained": achieved / fp8["sustained_tflops"], "peak_sustained": fp8["sustained_tflops"],
                "frac_of_bf16_x2": achieved / fp8_peak, "algorithmic_flops": flops, "ms_per_launch": idx_ms}
    else:
        achieved = idx_bytes / (idx_ms / 1000.0) / 1e9
        kname = "fp8 keys" if wl.key_fmt == I.KEY_FP8 else "mxfp4 keys"
        roof = {"kernel": f"indexer_kernel<{wl.rows_per_group}, {kname}>",
                "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_kind": peak_kind, "algorithmic_bytes": idx_bytes, "ms_per_launch": idx_ms,
                "timing": "back-to-back launches of the step's scorer calls in one CUDA graph, events at its ends",
                "ms_per_launch_event_nodes": idx_ms_events}
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            traffic = json.load(f).get(wl.name)
    # scorer, top-k (with page -> slot unless single pass, which launches it apart), sparse MLA;
    # decode with split rows adds the query prep and the merge; the histogram top-k of few long
    # rows runs as three launches
    launches_per_step = 3 + (1 if args.single_pass else 0) + (
        2 if (not prefill and P.sparse_mla_workspace_size(wl.num_rows, wl.heads, wl.k) > 0) else 0) + (
        2 if (not args.single_pass and P.topk_workspace_size(wl.num_rows, inp.max_ctx, wl.k) > 0) else 0)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3xe4m3->f32 (indexer), f16xf16->f32 (mla)", "data": "synthetic",
        "config": dsa_config(wl, copies, inp.idx_pool.numel() + inp.lat_pool.numel(), world, args.single_pass),
        "repeats_ms_per_step": [m / args.steps for m in rep_ms],
        "layer_hbm_gbs": layer_bytes / (ms_per_step / 1000.0) / 1e9,
        "layer_algorithmic_bytes": layer_bytes,
        "layer_frac_of_8tbs": layer_bytes / (ms_per_step / 1000.0) / 8e12,
        "roofline": dict(roof, traffic=traffic),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "launch": "one CUDA-graph replay per step between its copies" if e2e_graphs is not None
                else "eager launches between the copies"},
        "gpu_launches": launches_per_step * args.steps,
        "launch": {"multi-step": f"CUDA graphs of {16 * copies} consecutive steps (decode query prep on a "
                                 f"parallel branch beside the top-k); indexer timed after the timed loop by event nodes "
                                 f"around each scorer launch in a replay of the same steps "
                                 f"({len(samples)} launches sampled)",
                   "two-graphs": "CUDA-graph replay (indexer graph + rest-of-step graph), stream events between",
                   "eager": "eager launches, stream events around the indexer"}[graph_mode],
        "clocks": dict(clk.summary(h0, h2), window=f"the {REPEATS} timed regions and {h2 - h1:.2f} s of the "
                                                       f"same steps right after them"),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
