"""Throughput of attention with a learnable per-head sink, forward + backward.

One step = attn_sink_fwd + attn_sink_bwd (through the C ABI) over one batch of
the workload (default: the long batch, B=4, N=16384, H_q=64, H_kv=8, d=64,
causal, q scaled by 3, the largest single-GPU configuration).  Prints one
JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU float64 oracle, on host cores
  python bench.py --decode [--steps K] [--warmup W]   # the paged decode step
  python bench.py --record-traffic CSV --workload NAME [--traffic-scale X]
      # store the DRAM bytes of an ncu capture in profiles/dram_traffic.json

Timing: CUDA events on the launching stream around the fwd and bwd calls of
each step, and (recorded by the library on the same stream) around each launch
of the forward kernel and the backward main kernel for the roofline; a 256 MiB buffer is written between steps (outside the events) so
every step starts with a cold L2.  Under torchrun every rank runs its own
replica (no collective in the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from attention_learnable_head_gb300.inputs import WORKLOADS, make_case  # noqa: E402

METRIC = "attention-with-sinks fwd and bwd TFLOP/s on 1 GB300; % of dense-bf16 peak"
DET_METRIC = ("attention-with-sinks fwd and bitwise-reproducible bwd TFLOP/s on 1 GB300; "
              "% of dense-bf16 peak")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- counting
def visible_pairs(lengths, causal: bool, window: int) -> int:
    """Visible (query, key) pairs per query head, summed over the sequences."""
    total = 0
    for n in lengths:
        if not causal:
            total += n * n
        elif window <= 0:
            total += n * (n + 1) // 2
        else:
            w = min(window, n)
            total += w * (w + 1) // 2 + (n - w) * w
    return total


def forward_kernel(w) -> str:
    """The forward kernel the library launches for a workload: the
    sliding-window kernel when a causal window's items (128 / G tokens x the G
    query heads of a kv group) see at most 176 keys, else the tile kernel."""
    g = w.heads_q // w.heads_kv
    if w.causal and w.window > 0 and 128 % g == 0:
        cols = -(-(128 // g + w.window - 1) // 16) * 16
        if cols <= 176:
            return "attn_sink_fwd_band_kernel"
    return "attn_sink_fwd_kernel"


def algorithmic(w, lengths):
    """Algorithmic flops (fwd 4 d, bwd 10 d per pair and head) and minimum bytes."""
    pairs = visible_pairs(lengths, w.causal, w.window)
    d, hq, hkv = w.head_dim, w.heads_q, w.heads_kv
    t = sum(lengths)
    fwd_flops = 4.0 * d * hq * pairs
    bwd_flops = 10.0 * d * hq * pairs
    q_bytes, kv_bytes, lse_bytes = t * hq * d * 2, t * hkv * d * 2, t * hq * 4
    fwd_bytes = q_bytes + 2 * kv_bytes + q_bytes + lse_bytes
    bwd_bytes = (q_bytes + 2 * kv_bytes + q_bytes + q_bytes + lse_bytes      # q k v out dout lse
                 + q_bytes + 2 * kv_bytes + hq * 4)                          # dq dk dv dsink
    return dict(pairs=pairs, fwd_flops=fwd_flops, bwd_flops=bwd_flops, fwd_bytes=fwd_bytes,
                 bwd_bytes=bwd_bytes)


# the kernel's own code and the host code that picks its launch shape (grid,
# GQA split), both of which decide its DRAM traffic
KERNEL_SOURCES = {
    "attn_sink_fwd_kernel": ("fwd_kernel.cuh", "sm103_ptx.cuh", "attn_sink_api.cu"),
    "attn_sink_fwd_band_kernel": ("fwd_band_kernel.cuh", "fwd_kernel.cuh", "sm103_ptx.cuh",
                                  "attn_sink_api.cu"),
    "attn_sink_bwd_main_kernel": ("bwd_kernel.cuh", "sm103_ptx.cuh", "attn_sink_api.cu"),
}


def kernel_sources_hash(kernel: str) -> str:
    """sha256 (first 16 hex digits) of the code of the source files that define
    `kernel`: comments removed and whitespace collapsed, so that only a change
    of code counts."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "attention_learnable_head_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "dram_traffic.json")


def dram_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the ncu
    counters stored in profiles/dram_traffic.json (written by --record-traffic),
    or None when none were taken or the kernel's sources changed since (each
    entry carries their hash)."""
    if kernel not in KERNEL_SOURCES or not os.path.exists(TRAFFIC_JSON):
        return None
    with open(TRAFFIC_JSON) as f:
        entries = json.load(f).get("entries", [])
    want = kernel_sources_hash(kernel)
    for e in entries:
        if e["kernel"] == kernel and e["workload"] == workload:
            if e["sources_sha256"] != want:
                return None
            return float(e["dram_bytes_read"]) + float(e["dram_bytes_write"])
    return None


def record_traffic(csv_path: str, workload: str, scale: float, command: str):
    """Parse an ncu CSV (--csv, one row per launch and metric) and store, per
    kernel of KERNEL_SOURCES, the mean DRAM bytes read / written per launch,
    times `scale` (for a capture on a smaller case whose traffic grows in
    proportion to the work), with the kernel's current source hash."""
    import csv
    per = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if r]
    head = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    cols = rows[head]
    ki, mi, vi, ui = (cols.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value",
                                               "Metric Unit"))
    idi = cols.index("ID")
    mult = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    for r in rows[head + 1:]:
        name = r[ki].split("(")[0].split("::")[-1].strip()
        if name not in KERNEL_SOURCES or r[mi] not in ("dram__bytes_read.sum",
                                                       "dram__bytes_write.sum"):
            continue
        val = float(r[vi].replace(",", "")) * mult.get(r[ui], 1.0)
        per.setdefault(name, {}).setdefault(r[idi], {})[r[mi]] = val
    data = {"entries": []}
    if os.path.exists(TRAFFIC_JSON):
        with open(TRAFFIC_JSON) as f:
            data = json.load(f)
    for name, launches in per.items():
        rd = [m["dram__bytes_read.sum"] for m in launches.values()]
        wr = [m["dram__bytes_write.sum"] for m in launches.values()]
        entry = {"kernel": name, "workload": workload,
                 "dram_bytes_read": scale * sum(rd) / len(rd),
                 "dram_bytes_write": scale * sum(wr) / len(wr),
                 "launches": len(rd), "scale": scale, "command": command,
                 "sources_sha256": kernel_sources_hash(name)}
        data["entries"] = [e for e in data["entries"]
                           if not (e["kernel"] == name and e["workload"] == workload)]
        data["entries"].append(entry)
        print(json.dumps(entry))
    data["entries"].sort(key=lambda e: (e["workload"], e["kernel"]))
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling (200 ms) in the background during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.4)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle
def cpu_oracle_rates(w, case, budget_s: float, threads: int | None = None):
    """Time the CPU float64 oracle on whole query heads of the workload (all
    rows of every sequence): the forward (oracle_fwd) for about a third of
    ``budget_s`` and forward + backward (oracle_bwd, which recomputes the
    forward) for the rest, at least one head each.  Rates use the same
    algorithmic flops as the GPU line (fwd 4 d, bwd 10 d per visible pair)."""
    from oracle import oracle_bwd, oracle_fwd  # test infrastructure: only this leg runs it
    torch.set_num_threads(threads or os.cpu_count() or 1)
    cu = case.cu_seqlens
    pairs = visible_pairs(case.lengths, w.causal, w.window)
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, cu_seqlens_q=cu,
              cu_seqlens_k=cu)

    def timed(fn, budget):
        fn(heads=[0])                      # warm-up call (thread pool, allocator), untimed
        done, t0 = 0, time.perf_counter()
        while done < w.heads_q:
            fn(heads=[done])
            done += 1
            if time.perf_counter() - t0 >= budget:
                break
        return done, time.perf_counter() - t0

    nf, tf = timed(lambda heads: oracle_fwd(case.q, case.k, case.v, case.sink, heads=heads,
                                            **kw), budget_s / 3)
    nb, tb = timed(lambda heads: oracle_bwd(case.q, case.k, case.v, case.sink, case.dout,
                                            heads=heads, **kw), budget_s * 2 / 3)
    d = w.head_dim
    t_fwd_head, t_both_head = tf / nf, tb / nb
    t_bwd_head = t_both_head - t_fwd_head
    return dict(
        value=14.0 * d * pairs / t_both_head / 1e12, unit="TFLOP/s",
        fwd_value=4.0 * d * pairs / t_fwd_head / 1e12,
        # the backward's own share, where it stands clear of the timing noise
        bwd_value=(10.0 * d * pairs / t_bwd_head / 1e12
                   if t_bwd_head > 0.1 * t_both_head else None),
        cores=torch.get_num_threads(), kind="oracle", seconds=tf + tb,
        sample=(f"{w.name}: forward of query heads 0..{nf - 1} and forward+backward of query "
                f"heads 0..{nb - 1} of {w.heads_q}, all rows of every sequence, float64; "
                f"value = fwd+bwd, bwd_value = (fwd+bwd time - fwd time) per head"))


def cpu_baseline_line(w, case, budget_s: float):
    """The cpu_baseline object: the workload on every host core, plus the tiny
    workload on one thread."""
    res = cpu_oracle_rates(w, case, budget_s)
    res.pop("seconds", None)
    tw = WORKLOADS["tiny"]
    tiny = cpu_oracle_rates(tw, make_case(tw), 0.5, threads=1)
    tiny.pop("seconds", None)
    res["tiny_1_thread"] = tiny
    torch.set_num_threads(os.cpu_count() or 1)
    return res


def config_dict(w, lengths, ws: int) -> dict:
    """The `config` object of both arms' lines (identical for one workload)."""
    packed = w.is_varlen
    return {"workload": w.name, "batch": None if packed else len(lengths),
            "lengths": lengths if packed else None,
            "seq_len": None if packed else lengths[0], "heads_q": w.heads_q,
            "heads_kv": w.heads_kv, "head_dim": w.head_dim, "causal": w.causal,
            "window": w.window, "q_scale": w.q_mult, "parallelism": f"replicas x{ws}",
            "l2": "GPU arm: flushed between steps (256 MiB write outside the timed events); "
                  "inputs on the CPU arm live in host memory"}


# --------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device=None) -> list[float]:
    """Element-wise max of a list of floats over all ranks of the default
    process group (identity without one): a step is as long as its slowest rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_tflops(flops_per_rank: float, world_size: int, ms: float) -> float:
    """Throughput of the whole job: every rank processes flops_per_rank (weak
    scaling, replicas) in `ms`, the max over ranks."""
    return world_size * flops_per_rank / (ms * 1e-3) / 1e12


def count_launches(binding, fn) -> int:
    """Kernels libattn_sink launches during fn (the library's own launch counter)."""
    n0 = binding.attn_sink_launch_count()
    fn()
    return binding.attn_sink_launch_count() - n0


def run_reference(args, w, case):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    steps = []
    rates = []
    res = None
    for i in range(args.warmup + args.steps):
        res = cpu_oracle_rates(w, case, budget_s=args.ref_budget)
        if i >= args.warmup:
            steps.append(res["seconds"])
            rates.append(res["value"])
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, case.lengths, ws),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": res["cores"],
                         "kind": "oracle", "sample": res["sample"],
                         "fwd_value": res["fwd_value"], "bwd_value": res["bwd_value"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- decode
DECODE_METRIC = "paged decode: KV-cache GB/s read on 1 GB300; % of measured HBM copy bandwidth"


def decode_case(batch: int, cached: int, heads_q: int, heads_kv: int, page: int, seed: int):
    """Seeded serving-shaped decode inputs on the host: every sequence holds
    `cached` keys in pages of `page` keys, the pool's pages handed out in a
    random order (as an allocator that has been running a while would)."""
    g = torch.Generator().manual_seed(seed)
    per_seq = (cached + page - 1) // page
    n_pages = batch * per_seq
    kc = torch.randn(n_pages, page, heads_kv, 64, generator=g).to(torch.bfloat16)
    vc = torch.randn(n_pages, page, heads_kv, 64, generator=g).to(torch.bfloat16)
    table = torch.randperm(n_pages, generator=g).to(torch.int32).view(batch, per_seq)
    lens = torch.full((batch,), cached, dtype=torch.int32)
    q = torch.randn(batch, heads_q, 64, generator=g).to(torch.bfloat16)
    sink = torch.randn(heads_q, generator=g)
    return q, kc, vc, table, lens, sink


def run_decode(args):
    """One step = attn_sink_decode (one launch: the key-split kernel, whose last
    CTA per (sequence, kv head) merges the splits with the sink) for a batch of
    128 sequences with 8192 cached keys each, H 64/8, page 16.  The cache (2.1
    GB) is larger than L2, so no flush is needed between steps."""
    from attention_learnable_head_gb300 import binding
    from attention_learnable_head_gb300.build import build
    B, L, HQ, HKV, PAGE, SCALE = 128, 8192, 64, 8, 16, 0.125
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    host = decode_case(B, L, HQ, HKV, PAGE, seed=4242)
    q, kc, vc, table, lens, sink = (t.to(dev) for t in host)
    cache_bytes = 2 * B * L * HKV * 64 * 2
    alg_bytes = cache_bytes + table.numel() * 4 + q.numel() * 2 * 2 + HQ * B * 4
    step = lambda: binding.decode(q, kc, vc, table, lens, sink, softmax_scale=SCALE)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches = count_launches(binding, step)
    clocks = ClockSampler(0)
    clocks.start()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    clock = clocks.stop()
    st, code = binding.attn_sink_device_error()
    if st != 0 or code != 0:
        raise RuntimeError(f"device error word {code:#x} after the decode steps")
    ms = statistics.median(times)
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    peaks, src = load_peaks()
    line = {
        "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "decode_serving", "batch": B, "cached_keys": L, "heads_q": HQ,
                   "heads_kv": HKV, "head_dim": 64, "page_size": PAGE, "window": 0,
                   "l2": "inputs larger than L2 (2.1 GB of cache), no flush"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_note": f"{src} copy bandwidth; achieved = algorithmic bytes "
                                  f"(cache {cache_bytes} + q, out, lse, block table) / step time"},
        "gpu_launches": launches * args.steps, "gpu_launches_per_step": launches,
        "clocks": clock,
    }
    if not args.no_cpu_baseline:
        from oracle.decode import oracle_decode  # test infrastructure: only this leg runs it
        torch.set_num_threads(os.cpu_count() or 1)
        hq, hkc, hvc, htable, hlens, hsink = host
        done, t0 = 0, time.perf_counter()
        while done < B:
            idx = torch.tensor([done])
            oracle_decode(hq[idx], hkc, hvc, htable[idx], hlens[idx], hsink, scale=SCALE)
            done += 1
            if time.perf_counter() - t0 >= args.cpu_budget:
                break
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": done * (cache_bytes / B) / dt / 1e9, "unit": "GB/s",
            "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"decode_serving: sequences 0..{done - 1} of {B}, float64"}
    print(json.dumps(line), flush=True)


CHUNK_METRIC = ("sequence-parallel forward (key chunks + sink-aware merge) TFLOP/s on 1 GB300; "
                "% of dense-bf16 peak")


def run_chunks(args):
    """One step = the forward of a dense workload whose keys are cut into C
    equal chunks per sequence: C launches of attn_sink_fwd_chunk (each chunk
    attended without the sink, under the global causal / window mask through
    q_pos0 = -chunk start) and one attn_sink_merge (the C results combined
    with the sink counted once), i.e. the single-GPU half of sequence
    parallelism.  Throughput counts the forward's algorithmic flops, so it
    compares with the plain forward; the merge is set against the copy
    bandwidth.  After the timed steps the merged result is compared with one
    plain forward of the whole sequences."""
    from attention_learnable_head_gb300 import binding
    from attention_learnable_head_gb300.build import build
    w = WORKLOADS[args.workload]
    C = args.chunks
    if w.is_varlen or C < 1 or w.seqlen % (128 * C) != 0:
        raise SystemExit(f"--chunks {C}: needs a dense workload whose length is a multiple of "
                         f"128 x C ({w.name}: {w.seqlen})")
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = make_case(w)
    b, n = len(case.lengths), case.lengths[0]
    nc, hq, T = n // C, w.heads_q, b * n
    q = case.q.to(dev).view(b, n, hq, 64)
    k = case.k.to(dev).view(b, n, w.heads_kv, 64)
    v = case.v.to(dev).view(b, n, w.heads_kv, 64)
    sink = case.sink.to(dev)
    # each chunk's keys of every sequence, as their own dense tensors (what one
    # rank of a sequence-parallel group holds)
    ks = [k[:, c * nc:(c + 1) * nc].contiguous() for c in range(C)]
    vs = [v[:, c * nc:(c + 1) * nc].contiguous() for c in range(C)]
    kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale)
    pc = binding.make_params(q.shape, ks[0].shape, **kw)
    o_parts = torch.empty((C, b, n, hq, 64), dtype=torch.bfloat16, device=dev)
    r_parts = torch.empty_like(o_parts)
    l_parts = torch.empty((C, hq, T), dtype=torch.float32, device=dev)
    out, res = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
    fws = torch.empty(max(binding.attn_sink_fwd_workspace_size(pc), 1), dtype=torch.uint8,
                      device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        for c in range(C):
            st = binding.attn_sink_fwd_chunk(pc, -c * nc, q, ks[c], vs[c], None, None,
                                             o_parts[c], r_parts[c], l_parts[c], fws,
                                             fws.numel())
            if st:
                raise binding.AttnSinkError(st, "attn_sink_fwd_chunk")
        st = binding.attn_sink_merge(C, T, hq, 64, o_parts, r_parts, l_parts, sink, out, res,
                                     lse)
        if st:
            raise binding.AttnSinkError(st, "attn_sink_merge")

    binding.attn_sink_kernel_timing(True)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    launches = count_launches(binding, step)
    for kid in (binding.ATTN_SINK_KERNEL_FWD, binding.ATTN_SINK_KERNEL_MERGE):
        binding.attn_sink_kernel_time(kid)          # discard the untimed launches
    clocks = ClockSampler(0)
    clocks.start()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)                        # L2 flushed outside the events
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clock = clocks.stop()
    binding.attn_sink_kernel_timing(False)
    kt = {}
    for kid, per_step in ((binding.ATTN_SINK_KERNEL_FWD, C), (binding.ATTN_SINK_KERNEL_MERGE, 1)):
        st_k, ms_k, n_k = binding.attn_sink_kernel_time(kid)
        if st_k != 0 or n_k != per_step * args.steps:
            raise RuntimeError(f"kernel timing: status {st_k}, {n_k} launches")
        kt[kid] = ms_k / args.steps                  # per step (the C chunks summed)
    st, code = binding.attn_sink_device_error()
    if st != 0 or code != 0:
        raise RuntimeError(f"device error word {code:#x} after the chunked forward")
    # the same result as one plain forward over the whole sequences
    p_full = binding.make_params(q.shape, k.shape, **kw)
    out_f, res_f = torch.empty_like(q), torch.empty_like(q)
    lse_f = torch.empty_like(lse)
    ws_f = torch.empty(max(binding.attn_sink_fwd_workspace_size(p_full), 1), dtype=torch.uint8,
                       device=dev)
    if binding.attn_sink_fwd(p_full, q, k, v, sink, None, None, out_f, res_f, lse_f, ws_f,
                             ws_f.numel()):
        raise RuntimeError("plain forward for the comparison failed")
    full = out_f.float() + res_f.float()
    merged = out.float() + res.float()
    max_abs = float((merged - full).abs().max())
    lse_max_abs = float((lse - lse_f).abs().max())

    ms = statistics.median([e0.elapsed_time(e1) for e0, e1 in ev])
    alg = algorithmic(w, case.lengths)
    tf = alg["fwd_flops"] / (ms * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak, hbm = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
    fwd_ms, merge_ms = kt[binding.ATTN_SINK_KERNEL_FWD], kt[binding.ATTN_SINK_KERNEL_MERGE]
    fwd_tf = alg["fwd_flops"] / (fwd_ms * 1e-3) / 1e12
    # merge: C chunk outs and residuals (bf16) and lse (fp32) read, out, its
    # residual and lse written
    merge_bytes = C * T * hq * (64 * 2 * 2 + 4) + T * hq * (64 * 2 * 2 + 4) + hq * 4
    merge_gbs = merge_bytes / (merge_ms * 1e-3) / 1e9
    line = {
        "metric": CHUNK_METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(config_dict(w, case.lengths, 1), chunks=C, chunk_keys=nc),
        "roofline": {"kernel": "attn_sink_fwd_kernel (chunk mode)", "bound": "tensor",
                     "achieved": fwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": fwd_tf / peak,
                     "kernel_ms": fwd_ms, "launches_per_step": C, "traffic": None,
                     "peak_note": f"{src} dense bf16 burst; achieved = the forward's "
                                  f"algorithmic flops ({alg['fwd_flops']:.4g}) / the C chunk "
                                  f"launches' summed time"},
        "roofline_other": {"kernel": "attn_sink_merge_kernel", "bound": "hbm",
                           "achieved": merge_gbs, "peak": hbm, "unit": "GB/s",
                           "frac": merge_gbs / hbm, "kernel_ms": merge_ms, "traffic": None,
                           "algorithmic_bytes": merge_bytes,
                           "peak_note": f"{src} copy bandwidth; achieved = the bytes the merge "
                                        f"must move / kernel time"},
        "check": {"max_abs_vs_plain_forward": max_abs, "lse_max_abs_vs_plain_forward": lse_max_abs,
                  "note": "out + residual of the merged chunks against one attn_sink_fwd over "
                          "the whole sequences, every element"},
        "gpu_launches": launches * args.steps, "gpu_launches_per_step": launches,
        "clocks": clock,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = chunk_cpu_baseline(w, case, C, args.cpu_budget)
    print(json.dumps(line), flush=True)


def chunk_cpu_baseline(w, case, C: int, budget_s: float) -> dict:
    """The float64 oracle of the chunked forward and the merge (oracle_fwd_chunk,
    oracle_merge) on every host core, query head by query head of the first
    sequence until the budget is spent."""
    from oracle.chunk_merge import oracle_fwd_chunk, oracle_merge  # test infrastructure
    torch.set_num_threads(os.cpu_count() or 1)
    n = case.lengths[0]
    nc, group = n // C, w.heads_q // w.heads_kv
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, cu_seqlens_q=[0, n],
              cu_seqlens_k=[0, nc])
    done, t0 = 0, time.perf_counter()
    while done < w.heads_q:
        h, g = done, done // group
        qh = case.q[:n, h:h + 1]
        outs, lses = [], []
        for c in range(C):
            o, ls = oracle_fwd_chunk(qh, case.k[c * nc:(c + 1) * nc, g:g + 1],
                                     case.v[c * nc:(c + 1) * nc, g:g + 1], q_pos0=-c * nc, **kw)
            outs.append(o)
            lses.append(ls)
        oracle_merge(outs, lses, case.sink[h:h + 1])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    pairs = visible_pairs([n], w.causal, w.window)
    return {"value": 4.0 * w.head_dim * pairs * done / dt / 1e12, "unit": "TFLOP/s",
            "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"{w.name}: sequence 0, query heads 0..{done - 1} of {w.heads_q}, "
                      f"{C} key chunks and the merge, float64"}


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_full", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of CPU oracle work for the cpu_baseline leg")
    ap.add_argument("--ref-budget", type=float, default=6.0,
                    help="seconds of CPU oracle work per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu", action="store_true",
                    help="minimal run for a profiler: no e2e leg, no CPU baseline, no clock "
                         "sampling, no launch count")
    ap.add_argument("--decode", action="store_true",
                    help="time the paged decode step instead (one JSON line of its own)")
    ap.add_argument("--deterministic", action="store_true",
                    help="the same fwd+bwd step with the bitwise-reproducible backward "
                         "(attn_sink_bwd_deterministic); its own metric and config")
    ap.add_argument("--sink-bf16", action="store_true",
                    help="the same fwd+bwd step with the sink as a bf16 parameter whose "
                         "gradient accumulates (attn_sink_fwd_ex / attn_sink_bwd_ex flags); its "
                         "own metric and config")
    ap.add_argument("--chunks", type=int, default=0, metavar="C",
                    help="time the forward over C key chunks of every sequence plus the "
                         "sink-aware merge instead (one JSON line of its own)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="store the DRAM bytes per launch of an ncu capture (--csv with "
                         "dram__bytes_read.sum and dram__bytes_write.sum) of the workload "
                         "named by --workload in profiles/dram_traffic.json, and exit")
    ap.add_argument("--traffic-scale", type=float, default=1.0,
                    help="with --record-traffic: multiply the captured bytes (a capture of "
                         "a smaller case whose traffic grows in proportion)")
    ap.add_argument("--traffic-command", default="",
                    help="with --record-traffic: the ncu command line, stored with the entry")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic, args.workload, args.traffic_scale,
                       args.traffic_command)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.decode:
        run_decode(args)
        return
    if args.chunks:
        run_chunks(args)
        return

    w = WORKLOADS[args.workload]
    case = make_case(w)
    if args.impl == "reference":
        run_reference(args, w, case)
        return

    from attention_learnable_head_gb300 import binding
    from attention_learnable_head_gb300.build import build

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0 or ws == 1:
        build()
    if ws > 1:
        dist.barrier()
    binding.lib()

    lengths = case.lengths
    cu = torch.tensor(case.cu_seqlens, dtype=torch.int32, device=dev)
    q, k, v, dout = (t.to(dev) for t in (case.q, case.k, case.v, case.dout))
    sink = case.sink.to(dev)
    packed = w.is_varlen
    kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale)
    if not packed:
        b, n = len(lengths), lengths[0]
        q, dout = q.view(b, n, *q.shape[1:]), dout.view(b, n, *dout.shape[1:])
        k, v = k.view(b, n, *k.shape[1:]), v.view(b, n, *v.shape[1:])
    p = binding.make_params(q.shape, k.shape, num_seqs=len(lengths) if packed else None,
                            max_seqlen_q=max(lengths), max_seqlen_k=max(lengths), **kw)
    out = torch.empty_like(q)
    out_res = torch.empty_like(q)
    lse = torch.empty((w.heads_q, sum(lengths)), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if args.sink_bf16:
        # the sink as a bf16 training parameter; its gradient accumulates into dsink
        sink = sink.to(torch.bfloat16)
        dsink = torch.zeros_like(sink)
    else:
        dsink = torch.empty_like(sink)
    nws = binding.attn_sink_bwd_workspace_size(p)
    workspace = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
    fws = torch.empty(max(binding.attn_sink_fwd_workspace_size(p), 1), dtype=torch.uint8,
                      device=dev)
    cu_arg = cu if packed else None
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    if args.sink_bf16:
        def fwd_fn(*a):
            return binding.attn_sink_fwd_ex(a[0], binding.ATTN_SINK_FLAG_SINK_BF16, *a[1:])
    else:
        fwd_fn = binding.attn_sink_fwd

    def fwd():
        st = fwd_fn(p, q, k, v, sink, cu_arg, cu_arg, out, out_res, lse, fws, fws.numel())
        if st:
            raise binding.AttnSinkError(st, "attn_sink_fwd")

    det = args.deterministic
    bwd_fn = binding.attn_sink_bwd_deterministic if det else binding.attn_sink_bwd
    if args.sink_bf16:
        bwd_flags = (binding.ATTN_SINK_FLAG_SINK_BF16 | binding.ATTN_SINK_FLAG_ACCUMULATE_DSINK
                     | (binding.ATTN_SINK_FLAG_DETERMINISTIC if det else 0))

        def bwd_fn(*a):
            return binding.attn_sink_bwd_ex(a[0], bwd_flags, *a[1:])

    def bwd():
        st = bwd_fn(p, q, k, v, sink, cu_arg, cu_arg, out, out_res, lse, dout, dq, dk, dv, dsink,
                    workspace, workspace.numel())
        if st:
            raise binding.AttnSinkError(st, "attn_sink_bwd")
    timed_kernels = [binding.ATTN_SINK_KERNEL_FWD, binding.ATTN_SINK_KERNEL_BWD_MAIN]
    if det:
        timed_kernels.append(binding.ATTN_SINK_KERNEL_BWD_DQ)

    # per-kernel CUDA events (recorded by the library on the launching stream):
    # on from the warm-up so the event pool is filled before the timed region
    binding.attn_sink_kernel_timing(True)
    for _ in range(args.warmup):
        flush.fill_(1)
        fwd()
        bwd()
    torch.cuda.synchronize()
    launches_per_step = count_launches(binding, lambda: (fwd(), bwd()))
    for kid in timed_kernels:
        binding.attn_sink_kernel_time(kid)   # discard the warm-up launches

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if not args.ncu:
        sampler.start()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = binding.attn_sink_launch_count()
    wall0 = time.perf_counter()
    for i in range(n):
        flush.fill_(i & 0xFF)
        ev[i][0].record()
        fwd()
        ev[i][1].record()
        bwd()
        ev[i][2].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches_timed = binding.attn_sink_launch_count() - launches0
    binding.attn_sink_kernel_timing(False)
    kst = {}
    for kid in timed_kernels:
        st_k, ms_k, n_k = binding.attn_sink_kernel_time(kid)
        if st_k != 0 or n_k != n:
            raise RuntimeError(f"kernel timing: status {st_k}, {n_k} launches for {n} steps")
        kst[kid] = ms_k / n_k
    fwd_kernel_ms = kst[binding.ATTN_SINK_KERNEL_FWD]
    bwd_main_ms = kst[binding.ATTN_SINK_KERNEL_BWD_MAIN]
    bwd_dq_ms = kst.get(binding.ATTN_SINK_KERNEL_BWD_DQ, 0.0)
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    fwd_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    bwd_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    fwd_t, bwd_t = sum(fwd_ms) / n, sum(bwd_ms) / n
    step_ms = fwd_t + bwd_t
    step_ms, fwd_t, bwd_t, fwd_kernel_ms, bwd_main_ms, bwd_dq_ms = max_over_ranks(
        [step_ms, fwd_t, bwd_t, fwd_kernel_ms, bwd_main_ms, bwd_dq_ms], device=dev)

    # End to end through the C ABI with pinned host buffers: every step copies
    # its inputs in (q, k, v, dout, sink) and its results out (out, lse, dq, dk,
    # dv, dsink) inside the timed region.  As in a training loop, one step's
    # copies overlap its neighbours' compute: two device buffer sets, an upload,
    # a compute and a download stream, ordered by events.
    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, dout))
    hs = sink.cpu().pin_memory()
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory()
                 for t in (out, lse, dq, dk, dv, dsink)] for _ in range(2)]
    # the residual of out stays on the device (it only feeds the backward)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, hs))
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    # as many steps as the device-timed loop: the pipeline's fill (the first
    # upload) and drain (the last download) are paid once per run
    e2e_steps = 0 if args.ncu else max(3, n)
    dev_in = [(q, k, v, dout, sink),
              tuple(torch.empty_like(t) for t in (q, k, v, dout, sink))]
    dev_out = [(out, out_res, lse, dq, dk, dv, dsink),
               tuple(torch.empty_like(t) for t in (out, out_res, lse, dq, dk, dv, dsink))]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        bsel = i & 1
        qb, kb, vb, dob, sb = dev_in[bsel]
        ob, orb, lb, dqb, dkb, dvb, dsb = dev_out[bsel]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(cmp_done[bsel])      # step i-2 has read these inputs
            for d_, h in ((qb, hq), (kb, hk), (vb, hv), (dob, hdo), (sb, hs)):
                d_.copy_(h, non_blocking=True)
            in_ready[bsel].record(s_in)
        s_cmp.wait_event(in_ready[bsel])
        if i >= 2:
            s_cmp.wait_event(out_done[bsel])         # step i-2's results are on the host
        st = fwd_fn(p, qb, kb, vb, sb, cu_arg, cu_arg, ob, orb, lb, fws, fws.numel(), s_cmp)
        if st == 0:
            st = bwd_fn(p, qb, kb, vb, sb, cu_arg, cu_arg, ob, orb, lb, dob, dqb, dkb, dvb, dsb,
                        workspace, workspace.numel(), s_cmp)
        if st:
            raise binding.AttnSinkError(st, "e2e step")
        cmp_done[bsel].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[bsel])
            for h, d_ in zip(host_out[bsel], (ob, lb, dqb, dkb, dvb, dsb)):
                h.copy_(d_, non_blocking=True)
            out_done[bsel].record(s_out)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / max(e2e_steps, 1)], device=dev)[0]
    st, code = binding.attn_sink_device_error()
    if st != 0 or code != 0:
        raise RuntimeError(f"device error word {code:#x}")

    alg = algorithmic(w, lengths)
    flops = alg["fwd_flops"] + alg["bwd_flops"]
    value = whole_job_tflops(flops, ws, step_ms)
    fwd_tf = alg["fwd_flops"] / (fwd_t * 1e-3) / 1e12
    bwd_tf = alg["bwd_flops"] / (bwd_t * 1e-3) / 1e12
    peaks, src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    hbm = float(peaks["hbm_gbs"])
    # the dominant kernel is the longest of the forward kernel and the backward
    # main kernel (all five backward products; with the deterministic backward
    # four of them, S^T, dP^T, dV and dK, and the dQ kernel the other three,
    # S, dP recomputed and dQ); its achieved rate is the algorithmic flops of
    # its products (or the pass's minimum bytes) over its own launch time
    main_share = 0.8 if det else 1.0
    bwd_main_tf = main_share * alg["bwd_flops"] / (bwd_main_ms * 1e-3) / 1e12
    fwd_kernel_tf = alg["fwd_flops"] / (fwd_kernel_ms * 1e-3) / 1e12
    bwd_main_gbs = alg["bwd_bytes"] / (bwd_main_ms * 1e-3) / 1e9
    fwd_kernel_gbs = alg["fwd_bytes"] / (fwd_kernel_ms * 1e-3) / 1e9
    # which ceiling binds: the tensor cores, or HBM at the pass's arithmetic
    # intensity (the windowed layers)
    hbm_bound = (alg["bwd_flops"] / alg["bwd_bytes"]) * hbm / 1e3 < peak

    def roofline(kernel, tf, gbs, ms, bytes_alg, flops_alg, traffic=True):
        if hbm_bound:
            r = {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                 "frac": gbs / hbm, "tflops": tf, "tflops_frac_of_bf16_peak": tf / peak,
                 "peak_note": f"{src} copy bandwidth; achieved = the pass's minimum bytes "
                              f"({bytes_alg:.4g}) / kernel time"}
        else:
            r = {"kernel": kernel, "bound": "tensor", "achieved": tf, "peak": peak,
                 "unit": "TFLOP/s", "frac": tf / peak,
                 "frac_of_sustained": tf / float(peaks.get("bf16_tflops_sustained", peak)),
                 "hbm_gbs": gbs,
                 "peak_note": f"{src} dense bf16 burst; achieved = the algorithmic flops "
                              f"of the kernel's products ({flops_alg:.4g}) / kernel time"}
        # ncu counters are recorded for the default backward only
        r.update(kernel_ms=ms, traffic=dram_traffic(kernel, w.name) if traffic else None,
                 algorithmic_bytes=bytes_alg)
        return r

    rl_bwd = roofline("attn_sink_bwd_main_kernel", bwd_main_tf, bwd_main_gbs, bwd_main_ms,
                      alg["bwd_bytes"], main_share * alg["bwd_flops"], traffic=not det)
    rl_fwd = roofline(forward_kernel(w), fwd_kernel_tf, fwd_kernel_gbs, fwd_kernel_ms,
                      alg["fwd_bytes"], alg["fwd_flops"])
    ranked = [(bwd_main_ms, rl_bwd), (fwd_kernel_ms, rl_fwd)]
    if det:
        dq_tf = 0.6 * alg["bwd_flops"] / (bwd_dq_ms * 1e-3) / 1e12
        dq_gbs = alg["bwd_bytes"] / (bwd_dq_ms * 1e-3) / 1e9
        ranked.append((bwd_dq_ms, roofline("attn_sink_bwd_dq_kernel", dq_tf, dq_gbs, bwd_dq_ms,
                                           alg["bwd_bytes"], 0.6 * alg["bwd_flops"])))
    ranked.sort(key=lambda x: -x[0])
    dom, other = ranked[0][1], ranked[1][1]
    # Exponential-unit ceiling: one exp per visible pair and head in each pass,
    # ex2.approx.f32 at 32 results per SM clock (measured with a single-SM
    # probe), at the median SM clock sampled during the timed region.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    ex2_per_s = 32.0 * sms * mhz * 1e6
    sfu = {"ex2_per_sm_clock": 32, "sms": sms, "sm_mhz": mhz, "exp_per_s": ex2_per_s,
           "fwd_ceiling_tflops": ex2_per_s * 4 * w.head_dim / 1e12,
           "bwd_ceiling_tflops": ex2_per_s * 10 * w.head_dim / 1e12,
           "note": "fwd 4 d and bwd 10 d algorithmic flops per exponential"}
    config = config_dict(w, lengths, ws)
    metric = METRIC
    if det:
        config["backward"] = "deterministic"
        metric = DET_METRIC
    if args.sink_bf16:
        config["sink"] = "bf16 parameter, dsink accumulated"
        metric = metric.replace("TFLOP/s", "TFLOP/s (bf16 sink, accumulated dsink)", 1)
    line = {
        "metric": metric, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": n, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf, "fwd_ms": fwd_t, "bwd_ms": bwd_t,
        "frac_of_peak": value / peak, "fwd_frac_of_peak": fwd_tf / peak,
        "bwd_frac_of_peak": bwd_tf / peak, "peak_source": src,
        "roofline": dom,
        "roofline_other": other,
        **({"roofline_third": ranked[2][1]} if len(ranked) > 2 else {}),
        "sfu_ceiling": sfu,
        "e2e": None if args.ncu else {
            "value": whole_job_tflops(flops, ws, e2e_ms), "unit": "TFLOP/s",
            "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_timed,
        "gpu_launches_per_step": launches_per_step,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not args.ncu:
        line["cpu_baseline"] = cpu_baseline_line(w, case, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
