#!/usr/bin/env python
"""Sink-attention benchmark on one GB300 (or N replicas under torchrun).

Headline workload (one step = one pass of the whole decode path: scores, mask,
sink-initialised online softmax, P.V, split partials and their log-sum-exp
merge, bf16 output): decode over a contiguous KV cache, batch 64, one query
token per sequence, 64 query / 8 KV heads, head_dim 64, KV lengths uniform in
[1024, 8192], sinks ~N(0, 1). Metric: algorithmic KV bytes per second (every
visible K and V row once, plus q, out, lse and sinks).

Extras on the same run (reported, not the headline): varlen prefill (16
sequences, lengths uniform in [512, 4096], causal; full and window 128) and
4096-query chunked prefill over a 131072-token context in TFLOP/s of visible
(q, k) pairs (4 * 64 flops per pair), and paged decode (batch 256, contexts
uniform in [1024, 32768], 16-token pages; full and window 128) in GB/s, and
prefill against a 16-token paged cache (the chunked workload above, and 16
sequences with new chunks of 256..2048 tokens after 1k..32k cached ones) in
TFLOP/s, and 256 queries over a 131072-token context with the automatic
split-KV plan and without splits.

--impl reference times the float64 CPU oracle instead, on the same workload
and metric, one sequence (all heads) per step.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sink-attn decode KV GB/s & prefill TFLOP/s on 1 GB300, % of roofline"
WORKLOAD = ("decode_contig: batch 64, 1 query token each, 64 q / 8 kv heads, head_dim 64, "
            "bf16 KV lengths uniform in [1024, 8192], sinks ~N(0,1), full attention, "
            "split-KV with fused log-sum-exp merge")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="run one extra workload by name and print its numbers only "
                         "(for profiling one kernel)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ work ---

def decode_visible(lens, window):
    return [min(l, window) if window > 0 else l for l in lens]


def decode_bytes(case):
    """Algorithmic bytes of one decode call: every visible K and V row once
    (2 bytes per element, 1 for an fp8 cache), plus q, out (bf16), lse and
    sinks (fp32)."""
    elem = 1 if getattr(case, "kv_dtype", "bf16") == "fp8" else 2
    d = case.head_dim
    kv = sum(decode_visible(case.seqlens_k, case.window)) * case.hkv * d * elem * 2
    return kv + case.batch * case.hq * (d * 2 * 2 + 4) + case.hq * 4


def prefill_pairs(case):
    """Visible (query, key) pairs per head, summed over sequences."""
    tot = 0
    for lq, lk in zip(case.seqlens_q, case.seqlens_k):
        for i in range(lq):
            p = lk - lq + i
            hi = min(lk, p + 1) if case.causal else lk
            lo = max(0, p - case.window + 1) if case.window > 0 else 0
            tot += max(0, hi - lo)
    return tot


def prefill_io_bytes(case, kv_bytes):
    """The prefill's other roofline (HBM): Q and the visible K/V read once,
    out and lse written once, the sinks read. A short window makes the call
    HBM- or latency-bound rather than tensor-bound, so both are reported."""
    rows = sum(case.seqlens_q)
    return (rows * case.hq * case.head_dim * 2 * 2 + kv_bytes + rows * case.hq * 4
            + case.hq * 4)


def prefill_flops(case):
    return 4 * case.head_dim * prefill_pairs(case) * case.hq


# ---------------------------------------------------------------- clocks ---

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons around a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ distributed ---

def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if n > 1 or world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            import torch
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
        return rank, local, world, True
    return 0, 0, 1, False


def max_over_ranks(x, distributed, device="cpu"):
    if not distributed:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(distributed):
    if distributed:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ oracle leg ---

def oracle_decode_rate(case_cpu, seqs, reps=1):
    """Oracle (float64 CPU) time over the given sequences, all heads. Returns
    (GB/s of algorithmic bytes, seconds, threads)."""
    import torch

    import oracle
    q = case_cpu.q[seqs]
    lens = [case_cpu.seqlens_k[b] for b in seqs]
    kparts = [case_cpu.k[int(case_cpu.kv_indptr[b]):int(case_cpu.kv_indptr[b + 1])] for b in seqs]
    vparts = [case_cpu.v[int(case_cpu.kv_indptr[b]):int(case_cpu.kv_indptr[b + 1])] for b in seqs]
    k = torch.cat(kparts)
    v = torch.cat(vparts)
    from attention_learned_sinks_gb300 import synthetic as S
    indptr = S.offsets(lens)
    cu_q = torch.arange(0, len(seqs) + 1, dtype=torch.int32)
    threads = oracle.default_threads()
    oracle._lib()
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.attention(q, k, v, cu_q, indptr, hq=case_cpu.hq, hkv=case_cpu.hkv, head_dim=64,
                         sinks=case_cpu.sinks, causal=True, window=case_cpu.window,
                         scale=case_cpu.scale, nthreads=threads)
    dt = time.perf_counter() - t0
    nbytes = (sum(lens) * case_cpu.hkv * 64 * 4 + len(seqs) * case_cpu.hq * (64 * 4 + 4)
              + case_cpu.hq * 4) * reps
    return nbytes / dt / 1e9, dt, threads


def run_reference(args):
    """Float64 CPU oracle as the reference arm: rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch

    from attention_learned_sinks_gb300 import synthetic as S
    case = S.decode_contig(device="cpu")
    nb = case.batch
    for i in range(max(0, args.warmup)):
        oracle_decode_rate(case, [i % nb])
    t_total, bytes_total = 0.0, 0
    for i in range(args.steps):
        b = i % nb
        gbs, dt, threads = oracle_decode_rate(case, [b])
        t_total += dt
        bytes_total += gbs * dt * 1e9
    value = bytes_total / t_total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_total / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": "one sequence (all 64 heads) per step, "
                       "cycling through the 64-sequence batch"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle_threads(),
                             "kind": "oracle",
                             "sample": "one sequence of the decode_contig batch per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def oracle_threads():
    import oracle
    return oracle.default_threads()


# --------------------------------------------------------------- our arm ---

def time_calls(fn, reps, stream, flush=None):
    """Average device time of fn() over reps calls (CUDA events per call, L2
    optionally flushed before each call outside the timed interval)."""
    import torch
    times = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    return statistics.median(times)


def traffic_from_profile(name):
    """ncu DRAM bytes per launch recorded in profiles/<name>.md, valid only
    for the kernel source it was taken from (sha256 recorded there)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            if line.startswith("<!-- bench:"):
                rec = json.loads(line[len("<!-- bench:"):].split("-->")[0])
    if not rec:
        return None
    src = os.path.join(ROOT, "attention_learned_sinks_gb300", "csrc", rec["source"])
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if sha != rec.get("sha256"):
        return None
    return rec.get("traffic_bytes_per_launch")


def run_ours(args):
    import torch

    import attention_learned_sinks_gb300 as sa
    from attention_learned_sinks_gb300 import synthetic as S

    rank, local, world, distributed = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sa.load()
    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()
    if args.only:
        res = extras(sa, S, dev, stream, pk, pk_kind, only=args.only)
        if args.only not in res:
            raise SystemExit("unknown workload: " + args.only)
        print(json.dumps({"only": args.only, **res[args.only]}))
        return 0

    # ---- headline: contiguous decode, inputs resident in HBM ----
    case = S.decode_contig(device="cuda")
    kv_indptr = case.kv_indptr.to(dev)
    sinks = case.sinks.to(dev)
    out = torch.empty_like(case.q)
    lse = torch.empty((case.batch, case.hq), dtype=torch.float32, device=dev)
    need = sa.sinkattn_decode_workspace_size(case.batch, case.max_seqlen_k, case.hq, case.hkv)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)

    def step():
        sa.sinkattn_decode(case.q, case.k, case.v, kv_indptr=kv_indptr,
                           max_seqlen_k=case.max_seqlen_k, sinks=sinks, out=out, lse=lse,
                           workspace=ws)

    nbytes = decode_bytes(case)
    # the plan splits this workload: a counter-zeroing kernel precedes each decode
    launches_per_step = 2
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    # keep the clocks loaded for a moment before the timed region
    t_end = time.time() + 0.5
    while time.time() < t_end:
        step()
    barrier(distributed)
    torch.cuda.synchronize()
    # A few untimed steps queued in front of the start event: the device is
    # then busy when the timed region opens, so the host's marshalling and
    # launch latency of the first timed step is not counted.
    for _ in range(3):
        step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(distributed)
    clk = clocks.stop()
    elapsed = e0.elapsed_time(e1) / 1e3
    elapsed_max = max_over_ranks(elapsed, distributed, device=dev)
    per_step = elapsed_max / args.steps
    value = nbytes * world / per_step / 1e9
    achieved = nbytes / (elapsed / args.steps) / 1e9

    # ---- e2e through the public API from pinned host buffers ----
    hq_ = case.q.cpu().pin_memory()
    hk = case.k.cpu().pin_memory()
    hv = case.v.cpu().pin_memory()
    hind = case.kv_indptr.cpu().pin_memory()
    hs = case.sinks.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    dq, dk, dv = torch.empty_like(case.q), torch.empty_like(case.k), torch.empty_like(case.v)
    dind, ds = torch.empty_like(kv_indptr), torch.empty_like(sinks)

    def e2e_step():
        dq.copy_(hq_, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        dind.copy_(hind, non_blocking=True)
        ds.copy_(hs, non_blocking=True)
        sa.sinkattn_decode(dq, dk, dv, kv_indptr=dind, max_seqlen_k=case.max_seqlen_k, sinks=ds,
                           out=out, lse=lse, workspace=ws)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk, hv, hind, hs))
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 20))
    barrier(distributed)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_t = max_over_ranks(a.elapsed_time(b) / 1e3 / e2e_steps, distributed, device=dev)
    e2e_value = nbytes * world / e2e_t / 1e9
    del hk, hv, dk, dv

    peak_hbm = float(pk["hbm_gbs"])
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "kv_bytes_per_step": nbytes,
                   "l2": "inputs larger than L2 (%.2f GB of KV per step, no flush)" % (nbytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "split_plan": "auto (about 2 blocks per sequence and KV head)"},
        "roofline": {"kernel": "decode_kernel<contiguous> (after a 2 KB counter-zeroing kernel "
                               "it overlaps through programmatic dependent launch)",
                     "bound": "hbm", "achieved": achieved, "peak": peak_hbm, "unit": "GB/s",
                     "frac": achieved / peak_hbm, "peak_kind": pk_kind + " hbm_gbs",
                     "traffic": traffic_from_profile("decode_contig")},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }

    if not args.no_extra:
        line["extra"] = extras(sa, S, dev, stream, pk, pk_kind)

    if rank == 0 and not args.no_cpu_baseline:
        # the same batch on the host; one full pass, repeated until about 10 s
        # of CPU work has been timed (at most 100 passes)
        import dataclasses
        cpu_case = dataclasses.replace(case, q=case.q.cpu(), k=case.k.cpu(), v=case.v.cpu())
        seqs = list(range(cpu_case.batch))
        gbs, dt, threads = oracle_decode_rate(cpu_case, seqs)
        reps = 1
        if dt < 10.0:
            reps = min(100, max(1, int(10.0 / max(dt, 1e-3))))
            gbs, dt, threads = oracle_decode_rate(cpu_case, seqs, reps=reps)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": "the full 64-sequence batch, all heads, %d pass(es), "
                                          "%.1f s" % (reps, dt)}
    if rank == 0:
        print(json.dumps(line))
    if distributed:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def extras(sa, S, dev, stream, pk, pk_kind, only=None):
    """Prefill TFLOP/s and paged-decode GB/s on the other workloads."""
    import torch
    res = {}
    burst = float(pk["bf16_tflops"])
    hbm = float(pk["hbm_gbs"])
    # L2 flush between timed calls by READING 256 MB (twice the L2): a written
    # flush buffer would leave dirty lines whose write-back then lands inside
    # the next timed call (measured: +10 us on a 100 us decode)
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.sum()

    for name, mk, ns in (
            ("varlen_prefill", lambda: S.varlen_prefill(device="cuda"), 0),
            ("varlen_prefill_w128", lambda: S.varlen_prefill(window=128, device="cuda"), 0),
            ("varlen_prefill_d128", lambda: S.varlen_prefill_d128(device="cuda"), 0),
            ("varlen_prefill_g3", lambda: S.varlen_prefill_g3(device="cuda"), 0),
            ("chunked_prefill", lambda: S.chunked_prefill(device="cuda"), 0),
            ("long_context_prefill", lambda: S.long_context_prefill(device="cuda"), 0),
            ("long_context_prefill_unsplit", lambda: S.long_context_prefill(device="cuda"), 1)):
        if only is not None and name != only:
            continue
        c = mk()
        cq, ck = c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev)
        sk = c.sinks.to(dev)
        out = torch.empty_like(c.q)
        lse = torch.empty((c.q.shape[0], c.hq), dtype=torch.float32, device=dev)
        ws = torch.empty(sa.sinkattn_prefill_workspace_size(c.batch, c.q.shape[0], c.k.shape[0],
                                                            c.max_seqlen_q, c.max_seqlen_k, c.hq,
                                                            c.hkv, head_dim=c.head_dim,
                                                            window=c.window, num_splits=ns),
                         dtype=torch.uint8, device=dev)

        def call():
            sa.sinkattn_prefill(c.q, c.k, c.v, cq, ck, c.max_seqlen_q, c.max_seqlen_k, sinks=sk,
                                causal=c.causal, window=c.window, num_splits=ns, out=out, lse=lse,
                                workspace=ws)
        for _ in range(3):
            call()
        t = time_calls(call, 10, stream, flush)
        fl = prefill_flops(c)
        tokens = sum(c.seqlens_q)
        io = prefill_io_bytes(c, c.k.numel() * 2 + c.v.numel() * 2)
        res[name] = {"tflops": fl / t / 1e12, "ms": t * 1e3, "tokens_per_s": tokens / t,
                     "frac_of_bf16_peak": fl / t / 1e12 / burst,
                     "peak": burst, "peak_kind": pk_kind + " bf16_tflops (burst)",
                     "flops": fl, "num_splits": "auto" if ns == 0 else ns,
                     "io_bytes": io, "frac_of_hbm_peak": io / t / 1e9 / hbm}
        del c, out, lse, ws
        torch.cuda.empty_cache()

    # prefill against the paged cache: gather of the pages into contiguous
    # staging, then the same kernel; timed as one call (4 launches)
    for name, mk in (("paged_chunked_prefill", lambda: S.paged_chunked_prefill(device="cuda")),
                     ("paged_prefill_batch", lambda: S.paged_prefill_batch(device="cuda")),
                     ("paged_chunked_prefill_fp8",
                      lambda: S.paged_chunked_prefill_fp8(device="cuda"))):
        if only is not None and name != only:
            continue
        c = mk()
        cq, bt, sl = c.cu_seqlens_q.to(dev), c.block_table.to(dev), c.seqlens_k_t.to(dev)
        sk = c.sinks.to(dev)
        out = torch.empty_like(c.q)
        lse = torch.empty((c.q.shape[0], c.hq), dtype=torch.float32, device=dev)
        ws = torch.empty(sa.sinkattn_prefill_paged_workspace_size(c.batch, c.q.shape[0],
                                                                  c.max_seqlen_q, c.max_seqlen_k,
                                                                  c.hq, c.hkv, head_dim=c.head_dim,
                                                                  window=c.window),
                         dtype=torch.uint8, device=dev)

        fp8 = c.kv_dtype == "fp8"
        scales = {}
        if fp8:
            scales = {"k_scale": c.k_scale.to(dev), "v_scale": c.v_scale.to(dev)}

        def call():
            f = sa.sinkattn_prefill_paged_fp8 if fp8 else sa.sinkattn_prefill_paged
            f(c.q, cq, c.k_cache, c.v_cache, bt, sl, c.max_seqlen_q, c.max_seqlen_k, sinks=sk,
              causal=c.causal, window=c.window, out=out, lse=lse, workspace=ws, **scales)
        for _ in range(3):
            call()
        t = time_calls(call, 10, stream, flush)
        fl = prefill_flops(c)
        kv = sum(c.seqlens_k) * c.hkv * c.head_dim * 2 * (1 if fp8 else 2)
        io = prefill_io_bytes(c, kv)
        res[name] = {"tflops": fl / t / 1e12, "ms": t * 1e3,
                     "tokens_per_s": sum(c.seqlens_q) / t,
                     "frac_of_bf16_peak": fl / t / 1e12 / burst,
                     "peak": burst, "peak_kind": pk_kind + " bf16_tflops (burst)",
                     "flops": fl, "kv_bytes": kv,
                     "io_bytes": io, "frac_of_hbm_peak": io / t / 1e9 / hbm}
        del c, out, lse, ws
        torch.cuda.empty_cache()

    # backward of the varlen prefill (dq, dk, dv, dsinks), forward outputs
    # precomputed; algorithmic flops: 5 products of 2 * D per visible pair
    for name, w, d in (("varlen_backward", 0, 64), ("varlen_backward_w128", 128, 64),
                       ("varlen_backward_d128", 0, 128)):
        if only is not None and name != only:
            continue
        c = (S.varlen_prefill(window=w, device="cuda") if d == 64
             else S.varlen_prefill_d128(device="cuda"))
        cq, ck = c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev)
        sk = c.sinks.to(dev)
        out, lse = sa.sinkattn_prefill(c.q, c.k, c.v, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                       sinks=sk, causal=True, window=w)
        dout = S.bf16_normal(tuple(c.q.shape), 19, device="cuda")
        dq, dk, dv = torch.empty_like(c.q), torch.empty_like(c.k), torch.empty_like(c.v)
        dsk = torch.empty_like(sk)
        ws = torch.empty(sa.sinkattn_prefill_backward_workspace_size(c.batch, c.q.shape[0],
                                                                     c.k.shape[0], c.hq, c.hkv,
                                                                     c.head_dim),
                         dtype=torch.uint8, device=dev)

        def call():
            sa.sinkattn_prefill_backward(c.q, c.k, c.v, out, lse, dout, cq, ck, c.max_seqlen_q,
                                         c.max_seqlen_k, sinks=sk, causal=True, window=w, dq=dq,
                                         dk=dk, dv=dv, dsinks=dsk, workspace=ws)
        for _ in range(3):
            call()
        t = time_calls(call, 10, stream, flush)
        fl = 10 * c.head_dim * prefill_pairs(c) * c.hq
        res[name] = {"tflops": fl / t / 1e12, "ms": t * 1e3, "tokens_per_s": sum(c.seqlens_q) / t,
                     "frac_of_bf16_peak": fl / t / 1e12 / burst,
                     "peak": burst, "peak_kind": pk_kind + " bf16_tflops (burst)", "flops": fl}
        del c, out, lse, dout, dq, dk, dv, ws
        torch.cuda.empty_cache()

    # head_dim 128 (bf16 cache), and an fp8 e4m3 cache with per-KV-head scales:
    # contiguous (decode_contig's lengths) and paged (paged_decode's lengths,
    # 16-token pages)
    for name, mk in (("decode_contig_l2_flushed", lambda: S.decode_contig(device="cuda")),
                     ("decode_contig_d128", lambda: S.decode_contig_d128(device="cuda")),
                     ("decode_contig_fp8", lambda: S.decode_contig_fp8(device="cuda")),
                     ("paged_decode_fp8", lambda: S.make_decode(
                         "paged_decode_fp8", S.uniform_lengths(256, 1024, 32768, seed=4000), 64,
                         8, seed=4, sink_std=2.0, paged=True, device="cuda", kv_dtype="fp8"))):
        if only is not None and name != only:
            continue
        c = mk()
        sk = c.sinks.to(dev)
        fp8 = c.kv_dtype == "fp8"
        out = torch.empty_like(c.q)
        lse = torch.empty((c.batch, c.hq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, sa.sinkattn_decode_workspace_size(c.batch, c.max_seqlen_k, c.hq,
                                                                   c.hkv, c.head_dim)),
                         dtype=torch.uint8, device=dev)
        fn = sa.sinkattn_decode_fp8 if fp8 else sa.sinkattn_decode
        kw = dict(max_seqlen_k=c.max_seqlen_k, sinks=sk, out=out, lse=lse, workspace=ws)
        if fp8:
            kw.update(k_scale=c.k_scale.to(dev), v_scale=c.v_scale.to(dev))
        if c.paged:
            kw.update(block_table=c.block_table.to(dev), seqlens_k=c.seqlens_k_t.to(dev))
            kc, vc = c.k_cache, c.v_cache
        else:
            kw.update(kv_indptr=c.kv_indptr.to(dev))
            kc, vc = c.k, c.v

        def call():
            fn(c.q, kc, vc, **kw)
        for _ in range(3):
            call()
        t = time_calls(call, 10, stream, flush)
        nb = decode_bytes(c)
        res[name] = {"gbs": nb / t / 1e9, "ms": t * 1e3, "tokens_per_s": c.batch / t,
                     "frac_of_hbm_peak": nb / t / 1e9 / float(pk["hbm_gbs"]),
                     "kv_bytes": nb, "l2": "flushed before each call (256 MB read)"}
        del c, out, lse, ws
        torch.cuda.empty_cache()

    # paged_decode_b32: the paged workload's recipe with 32 sequences (about
    # 1.1 GB of KV, still well above L2): a profiling case only, run when
    # named with --only, never part of the default extras
    paged_cases = [("paged_decode", 0, 256), ("paged_decode_w128", 128, 256)]
    if only == "paged_decode_b32":
        paged_cases = [("paged_decode_b32", 0, 32)]
    for name, w, nbatch in paged_cases:
        if only is not None and name != only:
            continue
        c = S.paged_decode(window=w, device="cuda", batch=nbatch)
        bt, sl, sk = c.block_table.to(dev), c.seqlens_k_t.to(dev), c.sinks.to(dev)
        out = torch.empty_like(c.q)
        lse = torch.empty((c.batch, c.hq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, sa.sinkattn_decode_workspace_size(c.batch, c.max_seqlen_k, c.hq,
                                                                   c.hkv, window=w)),
                         dtype=torch.uint8, device=dev)

        def call():
            sa.sinkattn_decode(c.q, c.k_cache, c.v_cache, block_table=bt, seqlens_k=sl,
                               max_seqlen_k=c.max_seqlen_k, sinks=sk, window=w, out=out, lse=lse,
                               workspace=ws)
        for _ in range(3):
            call()
        t = time_calls(call, 10, stream, flush)
        nb = decode_bytes(c)
        res[name] = {"gbs": nb / t / 1e9, "ms": t * 1e3, "tokens_per_s": c.batch / t,
                     "frac_of_hbm_peak": nb / t / 1e9 / float(pk["hbm_gbs"]),
                     "kv_bytes": nb, "l2": "flushed before each call (256 MB read)"}
        del c, out, lse, ws
        torch.cuda.empty_cache()
    return res


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
