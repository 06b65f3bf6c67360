"""Benchmark: batched speculative-decoding verification on GB300.

One step = one spec_verify call (setup, row pass, filter/decide, draw) over the
B=256, k=15, V=151936 bfloat16 batch with top-k 50 / top-p 0.9 on both
distributions (2.41 GB of logits, far larger than the 129 MB L2, so no flush is
needed between steps).  Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Metric: verified rows per second (a verified row is one (request, position)
pair, sum_b (k_b + 1) per call), whole job over all ranks.  The roofline object
reports the row-pass kernel's achieved HBM bandwidth from the algorithmic bytes
(every target and draft logit once) over its CUDA-event duration.

--impl reference times the CPU oracle (the plain double-precision statement of
the method) on the host cores, on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank verifies its own independently seeded batch
(weak scaling, no data-path collective); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import signal
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "spec-verify rows/s and HBM GB/s vs ~8 TB/s peak at B=256,k=15,V=151936 bf16"
UNIT = "rows/s"
EVENT_EVERY = 8  # draft-sampler line: timed steps per row-pass event pair
ROWPASS_STEPS = 32  # verification line: steps timed for the row passes alone, after the K steps
INLINE_DRAW_V = 2048  # the library draws final tokens in the deciding warps up to this vocabulary
L2_BYTES = 129 * 1000 * 1000
FLUSH_BYTES = 512 << 20  # written between steps when the inputs fit in L2


def workload_desc(config, variant, batch=None):
    """The workload's name: its sizes and distributions, as the bench line
    reports them."""
    from speculative_decoding_verification_13_gb300 import workloads
    c = workloads.CONFIGS[config]
    B = c["B"] if batch is None else batch
    dt = "bf16" if c["dtype"].is_floating_point and c["dtype"].itemsize == 2 else "fp32"
    V = c["V"]
    if config in ("c1", "c2"):
        T = c["variants"][variant]
        mode = "greedy (T=0)" if T == 0 else f"temperature {T}"
        return (f"B={B} k={c['k']} V={V} {dt} logits, {mode}, draft = target + "
                f"N(0,{c['sigma']}^2), no filter")
    if config == "c3":
        return (f"B={B} k={c['k']} V={V} {dt} logits, temperature {c['temp']}, draft = target "
                f"+ N(0,{c['variants'][variant]}^2), no filter")
    if config == "c4":
        return (f"B={B} k={c['k']} V={V} {dt} logits, temperature 1, top-k {c['top_k']} + "
                f"top-p {c['top_p']} on p and q")
    if config == "c4p":
        return (f"B={B} k={c['k']} V={V} {dt} logits, temperature 1, top-p {c['top_p']} alone "
                f"on p and q (no top-k)")
    if config == "c5":
        return (f"B={B} ragged k~U{{1..15}} V={V} {dt} logits, 25% greedy else T~U[0.3,1.2], "
                f"draft noise sigma~U[0.3,2] per request, no filter")
    return config
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "rowpass_c4_traffic.json")
KERNEL_SOURCES = ["sv_internal.cuh", "sv_select.cuh", "sv_bigrow.cuh", "sv_rowpass.cu"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c4",
                    help="workload: c1..c5 (c4 = the headline), c4p = c4 with top-p alone")
    ap.add_argument("--variant", default=None,
                    help="c1/c2: t1|t0.7|greedy; c3: s0.5|s1|s2 (default: the first)")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the one-step comparison with the oracle after timing")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (small cases for profiling; not a bench line)")
    ap.add_argument("--path", choices=["verify", "sample", "kv", "lmhead"], default="verify",
                    help="verify: spec_verify (the headline); sample: the draft-side sampler "
                         "over the same workload's drafter rows")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, pg, device):
    """Max of a per-rank float over the process group: the step time of a
    weak-scaling run is the slowest rank's (nccl on the GPU, gloo in tests)."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "speculative_decoding_verification_13_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy read+write)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (profiling recipe, 6.8 TB/s)"


def recorded_traffic(rows, vocab):
    """DRAM bytes of a row-pass launch over `rows` bf16 rows of `vocab` logits,
    from the committed ncu summary: its per-row bytes (read + written) times
    the rows, only if it was taken on the current kernel source and on rows
    of the same length."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_hash") != kernel_hash() or d.get("vocab") != vocab:
        return None
    per_row = (d["dram_bytes_read_measured"] + d["dram_bytes_write_measured"]) / d["rows_measured"]
    return per_row * rows


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)],
                stdout=self.file, stderr=subprocess.DEVNULL, start_new_session=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            try:
                os.killpg(self.proc.pid, signal.SIGTERM)
            except Exception:
                pass
            self.proc.wait(timeout=10)
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(",") for l in self.file.read().splitlines() if l.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        sm.sort()
        med = sm[len(sm) // 2] if sm else None
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(batch_gpu, budget_s=12.0):
    """Oracle on the host cores over a bounded sample of the workload's
    requests (per-request parallel over all cores)."""
    import torch
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    B = batch_gpu.batch
    # calibrate on a small slice, then size the sample for ~budget_s of wall time
    n0 = min(B, max(cores, 8))
    sub = batch_gpu.requests(range(n0)).to("cpu")
    t0 = time.perf_counter()
    oracle.verify(sub.target, sub.draft, sub.draft_tokens, sub.k_per_req, sub.temperature,
                  sub.top_k, sub.top_p, sub.uniforms, threads=cores)
    dt = time.perf_counter() - t0
    n = int(min(B, max(n0, n0 * budget_s / max(dt, 1e-3))))
    sub = batch_gpu.requests(range(n)).to("cpu")
    # the sample is repeated (the whole batch may take well under the budget)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.verify(sub.target, sub.draft, sub.draft_tokens, sub.k_per_req, sub.temperature,
                      sub.top_k, sub.top_p, sub.uniforms, threads=cores)
        reps += 1
        dt = time.perf_counter() - t0
        if dt * cores >= budget_s * 3 or dt >= budget_s:
            break
    rows = sub.target_rows
    del sub
    torch.cuda.empty_cache()
    return {"value": reps * rows / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {B} requests ({rows} verified rows) x {reps}, "
                      f"per-request parallel over {cores} host threads, {dt:.2f} s wall"}


def run_reference(args, ws, rank):
    """The reference arm: the oracle as it stands, timed on the host cores."""
    if rank != 0:
        return
    import torch
    import oracle
    from speculative_decoding_verification_13_gb300 import workloads
    oracle.build()
    cores = os.cpu_count() or 1
    B = workloads.CONFIGS[args.config]["B"]
    variant = args.variant or next(iter(workloads.CONFIGS[args.config]["variants"]))
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    full = workloads.make_batch(args.config, variant, device=gen, batch=min(B, cores))
    # a bounded sample per step: one request per host thread, shrunk to a
    # single request when K + W steps would otherwise exceed ~150 s
    n = min(B, cores)
    sub = full.requests(range(n)).to("cpu")
    run = lambda: oracle.verify(sub.target, sub.draft, sub.draft_tokens, sub.k_per_req,
                                sub.temperature, sub.top_k, sub.top_p, sub.uniforms,
                                threads=cores)
    t0 = time.perf_counter()
    run()
    if (time.perf_counter() - t0) * (args.steps + args.warmup) > 150.0 and n > 1:
        n = 1
        sub = full.requests(range(n)).to("cpu")
    del full
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = sub.target_rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Zipf-plus-Gaussian logits, see workloads.py)",
        "config": {"workload": workload_desc(args.config, variant), "name": f"{args.config}:{variant}",
                   "sample_requests": n, "global_batch": B},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} requests ({sub.target_rows} verified rows) of the same "
                                   f"workload per step, per-request parallel over {cores} "
                                   f"threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_e2e(args, batch, v, acc, tok, stream, dev, pg):
    """Same metric through the public API from pinned host buffers: every step
    copies the step's inputs host->device and reads the results back."""
    import torch
    ws = pg.get_world_size() if pg else 1
    B, Rt = batch.batch, batch.target_rows
    filtered = batch.filters()[0] is not None
    names = ("target", "draft", "draft_tokens", "k_per_req", "temperature", "uniforms") + \
        (("top_k", "top_p") if filtered else ())
    host = {k: getattr(batch, k).to("cpu").pin_memory() for k in names}
    dbuf = {k: torch.empty_like(t, device=dev) for k, t in host.items()}
    acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
    tok_h = torch.empty(Rt, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = acc_h.numel() * 4 + tok_h.numel() * 4

    def e2e_step():
        for k_, t in host.items():
            dbuf[k_].copy_(t, non_blocking=True)
        a, o = v(dbuf["target"], dbuf["draft"], dbuf["draft_tokens"], dbuf["k_per_req"],
                 dbuf["temperature"], dbuf["uniforms"], dbuf.get("top_k"), dbuf.get("top_p"),
                 out_accept_len=acc, out_tokens=tok)
        acc_h.copy_(a, non_blocking=True)
        tok_h.copy_(o, non_blocking=True)

    for _ in range(2):
        e2e_step()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, pg, dev)
    del dbuf, host
    return {"value": ws * Rt / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "ms_per_step": e2e_ms}


SAMPLE_METRIC = "draft-sampler rows/s at B=256,k=15,V=151936 bf16 (top-k 50, top-p 0.9)"
SAMPLE_WORKLOAD = ("drafter rows of the B=256 k=15 V=151936 bf16 batch (3840 rows), "
                   "temperature 1, top-k 50 + top-p 0.9")


def run_sampler(args, ws, rank, local):
    """The draft-side sampler over the bench workload's drafter rows (one step
    = one spec_draft_sample call).  Same timing rules as the verifier's line;
    the roofline is the row pass over the drafter rows."""
    import torch
    import speculative_decoding_verification_13_gb300 as sv
    from speculative_decoding_verification_13_gb300 import build as cuda_build
    from speculative_decoding_verification_13_gb300 import workloads
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0:
        cuda_build.build()
    if pg:
        pg.barrier()
    sv.load_library()
    batch = workloads.make_batch(args.config, device=dev, seed_offset=rank, batch=args.batch)
    x, k, T = batch.draft, batch.k_per_req, batch.temperature
    tk, tp = batch.filters()
    R, V = x.shape
    g = torch.Generator(device=dev)
    g.manual_seed(1400 + rank)
    u = torch.rand(R, generator=g, device=dev)
    bytes_per_step = R * V * x.element_size()
    s = sv.DraftSampler(dev)
    tok = torch.empty(R, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda evs=None: s(x, k, T, u, tk, tp, out_tokens=tok, rowpass_events=evs)
    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    if s.error()[0] != 0:
        raise RuntimeError("device data error during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           if i % EVENT_EVERY == 0 else None for i in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(args.steps):
        call(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    step_ms = max_over_ranks(start.elapsed_time(end) / args.steps, pg, dev)
    timed = [e for e in evs if e is not None]
    rowpass_ms = sum(a.elapsed_time(b) for a, b in timed) / len(timed)
    clk = clocks.stop() if clocks else None
    e2e = None
    if not args.no_e2e:
        host = {n: t.to("cpu").pin_memory() for n, t in
                (("x", x), ("k", k), ("T", T), ("tk", tk), ("tp", tp), ("u", u))}
        dbuf = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
        tok_h = torch.empty(R, dtype=torch.int32).pin_memory()

        def e2e_step():
            for n, t in host.items():
                dbuf[n].copy_(t, non_blocking=True)
            o, _ = s(dbuf["x"], dbuf["k"], dbuf["T"], dbuf["u"], dbuf["tk"], dbuf["tp"],
                     out_tokens=tok)
            tok_h.copy_(o, non_blocking=True)

        for _ in range(2):
            e2e_step()
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, pg, dev)
        e2e = {"value": ws * R / (ms * 1e-3), "unit": "rows/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host.values()),
               "d2h_bytes_per_step": R * 4, "steps": args.e2e_steps, "ms_per_step": ms}
        del host, dbuf
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = os.cpu_count() or 1
        n = min(R, 1024)
        xs, us = x[:n].to("cpu"), u[:n].cpu()
        ks = torch.ones(n, dtype=torch.int32)  # rows are independent draws
        Ts, tks, tps = (t[:1].expand(n).cpu() for t in (T, tk, tp))
        reps = 0
        t0 = time.perf_counter()
        while True:  # repeated up to ~12 s of host-core work
            oracle.draft_sample(xs, ks, Ts, us, tks, tps, threads=cores)
            reps += 1
            dt = time.perf_counter() - t0
            if dt * cores >= 36.0 or dt >= 12.0:
                break
        cpu = {"value": reps * n / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"first {n} of {R} drafter rows x {reps}, parallel over {cores} "
                         f"host threads, {dt:.2f} s wall"}
    peak, peak_src = measured_peak()
    achieved = bytes_per_step / (rowpass_ms * 1e-3) / 1e9
    line = {
        "metric": SAMPLE_METRIC, "value": ws * R / (step_ms * 1e-3), "unit": "rows/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Zipf-plus-Gaussian logits, see workloads.py)",
        "config": {"workload": SAMPLE_WORKLOAD, "rows_per_step": R, "vocab": V,
                   "logit_bytes_per_step": bytes_per_step, "l2": "inputs larger than L2 "
                   "(1.17 GB of logits vs 129 MB), no flush",
                   "parallelism": f"replicas x{ws} (independent batches)"},
        "hbm_gbs": bytes_per_step / (step_ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "rowpass_kernel<bf16>", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": recorded_traffic(R, V) if x.dtype == torch.bfloat16 else None,
                     "traffic_source": "per-row DRAM bytes of the ncu capture of a B=64 "
                                       "verification launch (top-k rows, same V), x rows",
                     "peak_source": peak_src, "bytes_per_launch": bytes_per_step,
                     "launch_ms": rowpass_ms, "launches_timed": len(timed)},
        "e2e": e2e,
        "gpu_launches": (6 if tk is not None else 5) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


KV_METRIC = "KV-cache commit GB/s (read + write) after verifying B=256,k=15 (Qwen3-8B-class cache)"
KV_SHAPE = dict(layers=36, E=1024, S=16)  # 36 layers, 8 KV heads x 128, bf16, 16-token pages
KV_REPLICAS = 4
KV_GRAPH_STEPS = 20  # calls captured in the timed CUDA graph (a multiple of KV_REPLICAS)


def run_kv(args, ws, rank, local):
    """KV-cache commit after one verification of the bench workload: the
    accept lengths come from spec_verify on that batch; each request appends
    its last emitted token and its accepted drafts (36 layers x K and V x 1024
    bf16 = 147 KB per token) to a paged cache at a random offset in its page."""
    import torch
    import speculative_decoding_verification_13_gb300 as sv
    from speculative_decoding_verification_13_gb300 import build as cuda_build
    from speculative_decoding_verification_13_gb300 import workloads
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0:
        cuda_build.build()
    if pg:
        pg.barrier()
    sv.load_library()
    batch = workloads.make_batch(args.config, device=dev, seed_offset=rank, batch=args.batch)
    acc, _ = sv.verify(batch.target, batch.draft, batch.draft_tokens, batch.k_per_req,
                       batch.temperature, batch.uniforms, batch.top_k, batch.top_p)
    B, kmax = batch.batch, int(batch.k_per_req.max())
    layers, E, S = KV_SHAPE["layers"], KV_SHAPE["E"], KV_SHAPE["S"]
    g = torch.Generator(device=dev)
    g.manual_seed(1500 + rank)
    n0 = torch.randint(0, S, (B,), generator=g, device=dev, dtype=torch.int32)
    per_req = (S - 1 + kmax + 1 + S - 1) // S           # pages a request can touch
    n_pages = B * per_req
    table = torch.arange(n_pages, device=dev, dtype=torch.int32).view(B, per_req)
    table = table[:, torch.randperm(per_req, generator=g, device=dev)].contiguous()
    # KV_REPLICAS independent caches and speculative buffers, used in turn:
    # a step touches memory last used KV_REPLICAS - 1 steps (~500 MB) earlier,
    # so its reads come from HBM, not from the 129 MB L2
    caches = [torch.empty(n_pages, layers, 2, S, E, dtype=torch.bfloat16, device=dev)
              for _ in range(KV_REPLICAS)]
    specs = [torch.randn(B, kmax + 1, layers, 2, E, generator=g, device=dev).to(torch.bfloat16)
             for _ in range(KV_REPLICAS)]
    cache, spec = caches[0], specs[0]
    tokens = int((acc.clamp(min=-1) + 1).sum())
    bytes_per_step = 2 * tokens * layers * 2 * E * 2      # read and write
    # one kv_len array per call of a graph (KV_GRAPH_STEPS calls), all reset
    # to the starting lengths by one copy before the calls
    n0s = n0.repeat(KV_GRAPH_STEPS, 1)
    kv_lens = n0s.clone()
    stream = torch.cuda.current_stream(dev)

    def call(i):
        sv.kv_commit(caches[i % KV_REPLICAS], specs[i % KV_REPLICAS], acc, batch.k_per_req,
                     kv_lens[i], table)

    def calls():
        kv_lens.copy_(n0s)
        for i in range(KV_GRAPH_STEPS):
            call(i)
    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(max(1, args.warmup // KV_GRAPH_STEPS)):
        calls()
    torch.cuda.synchronize(dev)
    if sv.kv_commit_error(device=dev)[0] != 0:
        raise RuntimeError("KV commit data error during warm-up")
    # the host cost of one call through the Python binding (argument checks
    # and marshalling), which is of the order of the GPU's own time here
    t0 = time.perf_counter()
    for _ in range(3):
        calls()
    host_us = (time.perf_counter() - t0) / (3 * KV_GRAPH_STEPS) * 1e6
    torch.cuda.synchronize(dev)
    # the timed steps replay a CUDA graph of KV_GRAPH_STEPS calls (and the one
    # kv_len reset), so that the GPU's time is measured rather than the host's
    # issue rate
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        calls()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(graph):
        calls()
    replays = max(1, (args.steps + KV_GRAPH_STEPS - 1) // KV_GRAPH_STEPS)
    graph.replay()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for _ in range(replays):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize(dev)
    timed_steps = replays * KV_GRAPH_STEPS
    step_ms = max_over_ranks(start.elapsed_time(end) / timed_steps, pg, dev)
    if sv.kv_commit_error(device=dev)[0] != 0:
        raise RuntimeError("KV commit data error in the timed steps")
    clk = clocks.stop() if clocks else None
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    peak, peak_src = measured_peak()
    achieved = bytes_per_step / (step_ms * 1e-3) / 1e9
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        from oracle.kv import kv_commit as oracle_commit
        import numpy as np
        c_h = cache.view(torch.int16).cpu().numpy()
        s_h = spec.view(torch.int16).cpu().numpy()
        a_h, k_h, n_h, t_h = (t.cpu().numpy() for t in (acc, batch.k_per_req, n0, table))
        reps = 0
        t0 = time.perf_counter()
        while True:
            oracle_commit(s_h, a_h, k_h, n_h, t_h, c_h, S)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 3.0:
                break
        cpu = {"value": reps * bytes_per_step / dt / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"the whole step ({tokens} tokens) x {reps}, "
                                           f"one host thread, {dt:.2f} s wall"}
    line = {
        "metric": KV_METRIC, "value": ws * achieved, "unit": "GB/s", "n_gpus": ws,
        "steps": timed_steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (accept lengths from verifying the seeded bench batch; random K/V)",
        "timing": f"CUDA graph of {KV_GRAPH_STEPS} spec_kv_commit calls (one kv_len array "
                  f"each, all reset by one copy per graph), replayed {replays} times; host "
                  f"cost of one call through the Python binding {host_us:.1f} us",
        "config": {"workload": f"B={B} commits after k=15 verification, {tokens} tokens, "
                               f"{layers} layers x K,V x {E} bf16 per token, {S}-token pages",
                   "tokens_per_step": tokens, "bytes_per_step": bytes_per_step,
                   "l2": f"{KV_REPLICAS} cache / buffer replicas used in turn (each step's "
                         f"data last touched {KV_REPLICAS - 1} steps earlier), no flush",
                   "parallelism": f"replicas x{ws} (independent batches)"},
        "roofline": {"bound": "hbm", "kernel": "kv_copy_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": peak_src, "bytes_per_launch": bytes_per_step,
                     "note": "timed over whole calls (validation, copy, kv_len update)"},
        "e2e": None,
        "gpu_launches": 2 * timed_steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


LM_METRIC = "LM-head GEMM + verification statistics TFLOP/s (4096 target rows, V=151936, d=4096, bf16)"


def run_lmhead(args, ws, rank, local):
    """The target's LM head over the bench batch's target rows (B=256, k=15:
    4096 rows), V=151936, d=4096 (the hidden size of the pages' drafter code),
    with the verification statistics in the epilogue.  FLOPs = 2 M V d.  A
    torch.matmul of the same product (logits only, no statistics) is timed
    beside it for context."""
    import torch
    import speculative_decoding_verification_13_gb300 as sv
    from speculative_decoding_verification_13_gb300 import build as cuda_build
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0:
        cuda_build.build()
    if pg:
        pg.barrier()
    sv.load_library()
    M, V, d = (args.batch or 256) * 16, 151936, 4096
    g = torch.Generator(device=dev)
    g.manual_seed(1600 + rank)
    H = torch.randn(M, d, generator=g, device=dev).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=dev) / 16).to(torch.bfloat16)
    T = torch.ones(M, device=dev)
    tok = torch.randint(0, V, (M,), generator=g, device=dev, dtype=torch.int32)
    flops = 2.0 * M * V * d
    stream = torch.cuda.current_stream(dev)
    call = lambda: sv.lmhead_stats(H, W, T, tok)
    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    if sv.lmhead_stats_error(device=dev)[0] != 0:
        raise RuntimeError("LM-head kernel error during warm-up")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for _ in range(args.steps):
        call()
    end.record(stream)
    torch.cuda.synchronize(dev)
    step_ms = max_over_ranks(start.elapsed_time(end) / args.steps, pg, dev)
    clk = clocks.stop() if clocks else None
    # context: the same product by torch.matmul (cuBLAS), logits written out
    for _ in range(3):
        torch.matmul(H, W.T)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(max(1, args.steps // 2)):
        torch.matmul(H, W.T)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    mm_ms = e0.elapsed_time(e1) / max(1, args.steps // 2)
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except Exception:
        pass
    # a multi-millisecond kernel timed back to back: the sustained figure
    peak = peaks.get("bf16_tflops_sustained") or 1700.0
    peak_src = ("measured (MEASURED_PEAKS.json bf16_tflops_sustained, cuBLAS bf16)"
                if "bf16_tflops_sustained" in peaks else "fallback (profiling recipe, 1.7 PFLOP/s)")
    achieved = flops / (step_ms * 1e-3) / 1e12
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        from oracle.lmhead import lmhead_stats as oracle_stats
        n = 8
        Hs, Ws = H[:n].cpu(), W.cpu()
        t0 = time.perf_counter()
        oracle_stats(Hs, Ws, T[:n].cpu().numpy(), tok[:n].cpu().numpy())
        dt = time.perf_counter() - t0
        cpu = {"value": 2.0 * n * V * d / dt / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count() or 1, "kind": "oracle",
               "sample": f"{n} of {M} rows (float64 BLAS matmul and statistics), {dt:.2f} s wall"}
    line = {
        "metric": LM_METRIC, "value": ws * achieved, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random bf16 hidden states and unembedding)",
        "config": {"workload": f"M={M} rows, V={V}, d={d}, T=1, token per row",
                   "flops_per_step": flops, "l2": "unembedding 1.24 GB, larger than L2",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "tensor", "kernel": "lmhead_stats_kernel", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": peak_src, "flops_per_launch": flops,
                     "note": "timed over whole calls (GEMM kernel + combine kernel)"},
        "context": {"torch_matmul_tflops": flops / (mm_ms * 1e-3) / 1e12,
                    "torch_matmul_ms": mm_ms},
        "e2e": None,
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def required_bytes(batch):
    """Logit bytes the verification must read: every row of a sampled request,
    the target rows only of a greedy request (its draft rows are never read)."""
    k = batch.k_per_req.cpu().long()
    sampled = batch.temperature.cpu() > 0
    rows = int((k + 1).sum()) + int((k * sampled).sum())
    return rows * batch.vocab * batch.target.element_size(), rows


def parity_vs_oracle(batch, acc, tok, pq):
    """One verified step of the timed batch against the oracle (outside the
    timed region): counts of exempt requests and of mismatches, by the parity
    rule of oracle/compare.py."""
    import oracle
    from oracle.compare import compare
    import torch
    oracle.build()
    cpu = batch.to("cpu")
    t0 = time.perf_counter()
    o = oracle.verify(cpu.target, cpu.draft, cpu.draft_tokens, cpu.k_per_req, cpu.temperature,
                      cpu.top_k, cpu.top_p, cpu.uniforms, threads=os.cpu_count() or 1)
    dt = time.perf_counter() - t0
    g = dict(acc=acc.cpu().numpy(), tok=tok.cpu().numpy(),
             pq=pq[:batch.draft_rows].cpu().numpy() if pq is not None else None)
    dtn = "bfloat16" if cpu.target.dtype == torch.bfloat16 else "float32"
    rep = compare(cpu.k_per_req.numpy(), cpu.temperature.numpy(), cpu.vocab,
                  cpu.draft_tokens.numpy(), dtn, g, o, batch.name)
    out = rep.summary()
    out["pass"] = rep.ok()
    out["oracle_s"] = dt
    return out


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if args.path == "sample":
        run_sampler(args, ws, rank, local)
        return
    if args.path == "kv":
        run_kv(args, ws, rank, local)
        return
    if args.path == "lmhead":
        run_lmhead(args, ws, rank, local)
        return
    import torch
    import speculative_decoding_verification_13_gb300 as sv
    from speculative_decoding_verification_13_gb300 import build as cuda_build
    from speculative_decoding_verification_13_gb300 import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0:
        cuda_build.build()
    if pg:
        pg.barrier()
    sv.load_library()

    cfg = workloads.CONFIGS[args.config]
    variant = args.variant or next(iter(cfg["variants"]))
    batch = workloads.make_batch(args.config, variant, device=dev, seed_offset=rank,
                                 batch=args.batch)
    B, Rt, Rd, V = batch.batch, batch.target_rows, batch.draft_rows, batch.vocab
    bytes_formula = batch.logit_bytes()
    bytes_req, rows_req = required_bytes(batch)
    # the inputs of the small workloads fit in L2: flush it between steps
    flush = bytes_formula < 2 * L2_BYTES
    scratch = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    v = sv.Verifier(dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    tok = torch.empty(Rt, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    top_k, top_p = batch.filters()
    call = lambda evs=None: v(batch.target, batch.draft, batch.draft_tokens, batch.k_per_req,
                              batch.temperature, batch.uniforms, top_k, top_p,
                              out_accept_len=acc, out_tokens=tok, rowpass_events=evs)

    clocks = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    code = v.error()[0]
    if code != 0:
        raise RuntimeError(f"device data error {code} during warm-up")

    # timed region: K steps, no events between the kernels of a step (an
    # event recorded between two kernels ends the overlap of one kernel's
    # launch with the previous one's tail, about 8 us a step on the bench
    # workload).  With an L2 flush between steps each step is bracketed by its
    # own events (the flush is not timed).
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)] if flush else None
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(args.steps):
        if flush:
            scratch.fill_(i & 255)
            steps_ev[i][0].record(stream)
        call()
        if flush:
            steps_ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    if flush:
        step_ms = sum(a.elapsed_time(b) for a, b in steps_ev) / args.steps
    else:
        step_ms = start.elapsed_time(end) / args.steps
    # the streaming kernels alone: ROWPASS_STEPS more steps, each with events
    # recorded by the library right before and after its row passes
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(ROWPASS_STEPS)]
    for i in range(ROWPASS_STEPS):
        if flush:
            scratch.fill_(i & 255)
        call(evs[i])
    torch.cuda.synchronize(dev)
    timed = evs
    rowpass_ms = sum(a.elapsed_time(b) for a, b in timed) / len(timed)
    clk = clocks.stop() if clocks else None

    step_ms = max_over_ranks(step_ms, pg, dev)

    e2e = None if args.no_e2e else measure_e2e(args, batch, v, acc, tok, stream, dev, pg)
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    peak, peak_src = measured_peak()
    achieved = bytes_req / (rowpass_ms * 1e-3) / 1e9
    traffic = recorded_traffic(rows_req, V) \
        if batch.target.dtype == torch.bfloat16 and args.config in ("c4",) else None
    cpu = None
    parity = None
    if ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(batch)
    if ws == 1 and not args.no_parity:
        pq = torch.full((max(Rd, 1), 2), float("nan"), dtype=torch.float64, device=dev)
        a1, t1 = v(batch.target, batch.draft, batch.draft_tokens, batch.k_per_req,
                   batch.temperature, batch.uniforms, top_k, top_p, out_pq=pq)
        parity = parity_vs_oracle(batch, a1, t1, pq)
    dtype = "bf16" if batch.target.dtype == torch.bfloat16 else "f32"
    line = {
        "metric": METRIC,
        "value": ws * Rt / (step_ms * 1e-3),
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic (seeded Zipf-plus-Gaussian logits, see workloads.py)",
        "config": {"workload": workload_desc(args.config, variant, args.batch),
                   "name": f"{args.config}:{variant}",
                   "global_batch": ws * B, "per_gpu_batch": B,
                   "k": cfg["k"] if cfg["k"] is not None else "U{1..15}",
                   "vocab": V, "verified_rows_per_step": Rt,
                   "logit_rows_per_step": Rt + Rd, "logit_bytes_per_step": bytes_formula,
                   "required_logit_rows_per_step": rows_req,
                   "required_logit_bytes_per_step": bytes_req,
                   "l2": (f"inputs ({bytes_formula / 1e6:.1f} MB) fit in L2: a "
                          f"{FLUSH_BYTES >> 20} MB buffer is written before every step, "
                          f"outside the per-step events" if flush else
                          f"inputs larger than L2 ({bytes_formula / 1e9:.2f} GB of logits vs "
                          f"129 MB), no flush"),
                   "parallelism": f"replicas x{ws} (independent batches)"},
        "hbm_gbs": bytes_req / (step_ms * 1e-3) / 1e9,
        "hbm_gbs_formula": bytes_formula / (step_ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": f"rowpass_kernel<{dtype}>", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": peak_src,
                     "bytes_per_launch": bytes_req, "launch_ms": rowpass_ms,
                     "launches_timed": len(timed)},
        "e2e": e2e,
        # setup, row pass, [threshold row pass], filter / decide, [draw pass,
        # locate]: vocabularies up to INLINE_DRAW_V take their draws in the
        # decide warps, without the last two launches
        "gpu_launches": (3 + (top_k is not None) + (2 if V > INLINE_DRAW_V else 0)) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "parity": parity,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
