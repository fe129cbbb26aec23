#!/usr/bin/env python
"""Benchmark of one MSA training step on GB300.

A step is one pass of the whole hot path over one batch: proxy scoring with
block max-pool and top-k selection (msa_proxy_select), block-sparse attention
forward (msa_fwd) and backward with the fused proxy-KL gradient (msa_bwd), all
through the C ABI of libmsa.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 128k|512k|1m|varlen|tiny]
                    [--impl ours|reference] [--no-dense] [--no-cpu-baseline] [--no-configs]
                    [--only-select]

Prints one JSON line (rank 0).  `value` is the effective TFLOP/s of the step
on the headline workload (128k tokens unless --workload says otherwise):
14*d FLOPs per (query head, key) pair inside the selection mask (4d forward,
10d backward; the diagonal block counts only its causal keys), divided by the
measured step time; proxy scoring is not counted but its time is.  Inputs are
synthetic (seeded, see synth/) and resident in HBM when the timed region
starts; they are larger than L2, so no flush is needed between steps.
`e2e` is the same metric with the inputs in pinned host memory, copied to the
device every step inside the timed region, and the step's results (O, LSE,
the five gradients, the loss) copied back to pinned host memory, also inside
it (HostInputStep: the copies overlap the kernels on two copy streams).
`per_config` repeats the measurement for every workload of the metric's range
(1k tiny, 32k varlen, 128k, 512k, 1M), each with the dense SDPA comparator and
the fp64 CPU oracle timed on the host cores (every row for the tiny and varlen
workloads, a seeded sample of rows for the others).
With N > 1 (torchrun), every rank runs an independent replica on its own GPU
(the path has no exchange step); the aggregate counts all ranks' work over the
slowest rank's time; per_config is measured on rank 0's GPU only.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MSA fwd+bwd effective TFLOPS (selected blocks) & tokens/s at 128k–1M, 1 GB300"
UNIT = "TFLOP/s"


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
# work accounting (host arithmetic on the document lengths)
# ---------------------------------------------------------------------------
def work_counts(w) -> dict:
    """Pair, slot and block counts of one step, from the document lengths."""
    B, K = w.block, w.top_k
    pairs = 0            # (query token, key) pairs inside the mask, per query head
    rowslots = 0         # (token, selected block) pairs, per query head
    causal = 0           # causal (query, key) pairs per KV group (proxy scoring)
    nblocks = 0
    for L in w.doc_lengths:
        i = np.arange(L, dtype=np.int64)
        j, r = i // B, i % B
        pairs += int(np.sum(np.minimum(j, K - 1) * B + r + 1))
        rowslots += int(np.sum(np.minimum(j, K - 1) + 1))
        causal += int(L) * (int(L) + 1) // 2
        nblocks += (int(L) + B - 1) // B
    return dict(pairs=pairs, rowslots=rowslots, causal=causal, nblocks=nblocks)


def flops_effective(w, c) -> float:
    return 14.0 * w.d * w.hq * c["pairs"]


def kernel_models(w, c) -> dict:
    """Algorithmic work per launch of the three block kernels.

    select (tensor-bound): 2*dp FLOPs per causal (query, key) pair per group.
    fwd (HBM-bound): per (token, head, slot): gathered q row (2d B), partial O
        row written as int16 (2d B) with its lse and scale (8 B); per (group,
        block): K and V tiles (2*128*2d B).
    bwd (HBM-bound): per (token, head, slot): q and dO rows (4d B), fp32 dQ
        partial (4d B), lse and D (8 B); per (token, group, slot): q_p row and
        proxy scalars (2dp + 13 B);
        per (group, block): K, V reads (4*128*d B), dK, dV writes (8*128*d B),
        dk_p write (4*128*dp B).
    """
    d, dp, hq, hkv = w.d, w.dp, w.hq, w.hkv
    rs = c["rowslots"] * hq
    ts = c["rowslots"] * hkv
    blk = c["nblocks"] * hkv
    return {
        1: dict(name="k_select", bound="tensor", work=2.0 * dp * hkv * c["causal"], unit="TFLOP/s"),
        2: dict(name="k_fwd", bound="hbm",
                work=rs * (4.0 * d + 8) + blk * (4.0 * 128 * d), unit="GB/s"),
        3: dict(name="k_bwd", bound="hbm",
                work=rs * (8.0 * d + 8) + ts * (2.0 * dp + 13) +
                blk * (4.0 * 128 * d + 8.0 * 128 * d + 4.0 * 128 * dp), unit="GB/s"),
    }


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = f"/tmp/msa_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return dict(sm_mhz=float(np.median(sm)) if sm else None,
                    sm_max_mhz=float(max(mx)) if mx else None,
                    reasons=sorted(reasons), samples=len(sm))


# ---------------------------------------------------------------------------
# ncu traffic recorded under profiles/ (null once the kernel source changed)
# ---------------------------------------------------------------------------
def kernel_source_sha(name: str) -> str:
    f = {"k_select": "k_select.cu", "k_fwd": "k_fwd.cu", "k_bwd": "k_bwd.cu"}[name]
    h = hashlib.sha256()
    for part in (f, "ptx.cuh", "msa_internal.cuh"):
        with open(os.path.join(ROOT, "block_sparse_attention_proxy_gb300", "csrc", part), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str, workload: str):
    """dram read+write bytes per launch from profiles/<kernel>_<workload>.md,
    if that summary was taken on the current source of the kernel."""
    path = os.path.join(ROOT, "profiles", f"{name}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m1 = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    m2 = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
    if not m1 or not m2 or m2.group(1) != kernel_source_sha(name):
        return None
    return float(m1.group(1))


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:  # host-only runs of the rank logic (CPU tests)
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: the aggregate throughput divides every rank's
    units by it."""
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_of(w, world: int = 1) -> dict:
    """The `config` object of the JSON line (identical in both arms)."""
    return dict(workload=f"{w.name}: {w.total_tokens} tokens in {w.num_docs} doc(s), "
                         f"Hq={w.hq} Hkv={w.hkv} d={w.d} dp={w.dp} block={w.block} "
                         f"top-k={w.top_k}" + (", rank-8 structured k/k_p" if w.structured else ""),
                tokens=w.total_tokens, l2="inputs larger than L2 (no flush)",
                parallelism="replicas" if world > 1 else "single GPU")


def make_device_inputs(w) -> dict:
    """Seeded inputs on the device: drawn on the CPU for the small workloads (so
    a CPU process can redraw the very same tensors), on the GPU for the rest."""
    if w.total_tokens <= 65536:
        return {k: v.cuda() for k, v in synth.make_inputs(w, device="cpu").items()}
    return synth.make_inputs(w, device="cuda")


def dense_sdpa(w, inp, steps=2, warmup=1, warm_tokens=None) -> dict:
    """torch SDPA (library backend) causal GQA fwd+bwd at the same shapes.

    Backends are tried in order: cuDNN with native GQA, cuDNN with K/V
    expanded to every query head, torch's flash kernel, then torch's default
    choice; the first that runs is timed.  warm_tokens: warm up on a prefix of
    that many tokens instead of the full batch (long sequences)."""
    from torch.nn.attention import SDPBackend, sdpa_kernel

    cu = inp["cu_seqlens"].tolist()
    qs = inp["q"].transpose(0, 1).unsqueeze(0)
    ks = inp["k"].transpose(0, 1).unsqueeze(0)
    vs = inp["v"].transpose(0, 1).unsqueeze(0)
    dos = inp["dO"].transpose(0, 1).unsqueeze(0)
    G = w.hq // w.hkv
    attempts = ((SDPBackend.CUDNN_ATTENTION, True, "cuDNN, native GQA"),
                (SDPBackend.CUDNN_ATTENTION, False, "cuDNN, K/V expanded per query head"),
                (SDPBackend.FLASH_ATTENTION, True, "flash (torch), native GQA"),
                (None, True, "torch default choice, native GQA"))
    errors = []
    for backend, native, label in attempts:
        def one(limit=None):
            spans = list(zip(cu[:-1], cu[1:]))
            if limit is not None:
                spans = [(spans[0][0], min(spans[0][1], spans[0][0] + limit))]
            for a, b in spans:
                q = qs[:, :, a:b].detach().requires_grad_(True)
                k = ks[:, :, a:b].detach().requires_grad_(True)
                v = vs[:, :, a:b].detach().requires_grad_(True)
                kk, vv = (k, v) if native else (k.repeat_interleave(G, 1), v.repeat_interleave(G, 1))
                o = torch.nn.functional.scaled_dot_product_attention(
                    q, kk, vv, is_causal=True, scale=1.0, enable_gqa=native and G > 1)
                o.backward(dos[:, :, a:b])

        try:
            ctx = sdpa_kernel(backend) if backend is not None else contextlib.nullcontext()
            with ctx:
                for _ in range(warmup):
                    one(warm_tokens)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(steps):
                    one()
                e1.record()
                torch.cuda.synchronize()
        except Exception as ex:  # the comparator is optional context
            errors.append(f"{label}: {type(ex).__name__}: {str(ex)[:120]}")
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            continue
        ms = e0.elapsed_time(e1) / steps
        dense_pairs = sum(L * (L + 1) // 2 for L in w.doc_lengths) * w.hq
        fl = 14.0 * w.d * dense_pairs
        torch.cuda.empty_cache()
        return dict(impl=f"torch.nn.functional.scaled_dot_product_attention, causal, {label}",
                    ms_per_step=round(ms, 3), tflops=round(fl / ms / 1e9, 2),
                    tokens_per_s=round(w.total_tokens / ms * 1e3, 1), steps=steps,
                    warmup=warmup, warm_tokens=warm_tokens, skipped=errors or None)
    return dict(unavailable="; ".join(errors)[:400])


class _Rows:
    """Rows t of a [T, ...] device tensor copied to the host (the oracle reads
    q, dO and q_p only at the sampled rows)."""

    def __init__(self, dev, rows):
        self.rows = {int(t): dev[int(t)].to("cpu") for t in rows}

    def __getitem__(self, t):
        return self.rows[int(t)]


def cpu_baseline(w, inp, n_rows: int, seed: int) -> dict:
    """The fp64 oracle as it stands, on a seeded sample of query rows (every
    head and group of each row, forward and backward incl. its dK/dV/dk_p
    contributions), on this host's cores.  The oracle reads the key-side
    tensors up to each row; those are copied to the host once (k_p upcast to
    fp64 once, exactly, since every row reads its whole prefix)."""
    from oracle import OracleParams, row_reference

    prm = OracleParams(w.hq, w.hkv, w.d, w.dp, w.top_k)
    rows = synth.sample_rows(w.total_tokens, n_rows, seed + 1000).tolist()
    cpu = dict(cu_seqlens=inp["cu_seqlens"].to("cpu"), k=inp["k"].to("cpu"), v=inp["v"].to("cpu"),
               k_p=inp["k_p"].to("cpu").double().numpy())
    for n in ("q", "dO", "q_p"):
        cpu[n] = _Rows(inp[n], rows)
    cu = cpu["cu_seqlens"].tolist()
    t0 = time.perf_counter()
    pairs = 0
    for t in rows:
        row_reference(cpu, prm, int(t), contributions=True)
        a = max(x for x in cu[:-1] if x <= t)
        i = t - a
        pairs += min(i // 128, w.top_k - 1) * 128 + i % 128 + 1
    dt = time.perf_counter() - t0
    fl = 14.0 * w.d * w.hq * pairs
    return dict(value=round(fl / dt / 1e12, 6), unit=UNIT, cores=torch.get_num_threads(),
                kind="oracle",
                sample=f"{len(rows)} seeded query rows of the {w.name} workload (all heads and "
                       f"groups, fwd+bwd); {dt:.1f} s wall",
                seconds=round(dt, 2), tokens_per_s=round(len(rows) / dt, 3))


def _oracle_all_rows(names, threads, queue):
    """Child process (spawned): the fp64 oracle on every row of the named small
    workloads, whose inputs it redraws on the CPU from the same seeds."""
    torch.set_num_threads(threads)
    from oracle import OracleParams, msa_reference

    for name in names:
        w = synth.workload(name)
        inp = synth.make_inputs(w, device="cpu")
        c = work_counts(w)
        t0 = time.perf_counter()
        msa_reference(inp, OracleParams(w.hq, w.hkv, w.d, w.dp, w.top_k), with_grads=True)
        dt = time.perf_counter() - t0
        fl = flops_effective(w, c)
        queue.put((name, dict(value=round(fl / dt / 1e12, 6), unit=UNIT, cores=threads,
                              kind="oracle",
                              sample=f"every row of the {name} workload ({w.total_tokens} tokens, "
                                     f"all heads and groups, fwd+bwd); {dt:.1f} s wall",
                              seconds=round(dt, 2), tokens_per_s=round(w.total_tokens / dt, 3))))


def time_steps(step, inp, K, W, world, profile=True):
    """W untimed steps, then K steps timed with CUDA events between barriers;
    per-call and per-block-kernel times from events recorded on the stream."""
    import block_sparse_attention_proxy_gb300 as m

    for _ in range(W):
        step(inp)
    torch.cuda.synchronize()
    if m.msa_get_device_status() != 0:
        raise RuntimeError(f"device status {m.msa_last_status_word():#x} after warm-up")
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    kev = [[(E(), E()) for _ in range(3)] for _ in range(K)]
    call_ev = [[E() for _ in range(4)] for _ in range(K)]
    for pairs_ in kev:  # torch creates the CUDA event handles on first record
        for a_, b_ in pairs_:
            a_.record()
            b_.record()
    torch.cuda.synchronize()
    t0, t1 = E(), E()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = m.msa_launch_count()
    t0.record()
    for i in range(K):
        if profile:
            for kid in range(3):
                m.msa_set_profile_events(kid + 1, *kev[i][kid])
        call_ev[i][0].record()
        step.select(inp)
        call_ev[i][1].record()
        step.forward(inp)
        call_ev[i][2].record()
        step.backward(inp)
        call_ev[i][3].record()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    launches = m.msa_launch_count() - launches0
    clk = clocks.stop()
    for kid in range(3):
        m.msa_set_profile_events(kid + 1, None, None)
    st = m.msa_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {m.msa_last_status_word():#x} in the timed region")
    ms_local = t0.elapsed_time(t1) / K
    kern_ms = ({kid + 1: sum(kev[i][kid][0].elapsed_time(kev[i][kid][1]) for i in range(K)) / K
                for kid in range(3)} if profile else {})
    calls = {n: sum(call_ev[i][a].elapsed_time(call_ev[i][a + 1]) for i in range(K)) / K
             for n, a in (("select", 0), ("fwd", 1), ("bwd", 2))}
    return ms_local, kern_ms, calls, launches, clk


# steps, warm-up, dense-comparator steps, CPU-oracle rows (None: every row, in
# the spawned process) of the per-config records; the headline workload uses
# the command line's steps and warm-up
PER_CONFIG = {"tiny": (10, 3, 5, None), "varlen": (10, 3, 3, None), "128k": (5, 3, 1, 64),
              "512k": (3, 3, 1, 32), "1m": (3, 3, 1, 24)}


def measure_config(name, peaks, args, cpu_rows, dense_steps, K, W, world=1) -> dict:
    """One workload: step time, kernel split, dense comparator, CPU oracle."""
    from block_sparse_attention_proxy_gb300.step import MSAStep, params_for

    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats()
    w = synth.workload(name)
    c = work_counts(w)
    inp = make_device_inputs(w)
    prm = params_for(inp["cu_seqlens"].tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k)
    step = MSAStep(prm)
    ms, kern_ms, calls, launches, clk = time_steps(step, inp, K, W, world)
    fl = flops_effective(w, c)
    models = kernel_models(w, c)
    rec = dict(workload=config_of(w)["workload"], tokens=w.total_tokens, steps=K, warmup=W,
               ms_per_step=round(ms, 3), tflops=round(fl / ms / 1e9, 3),
               tokens_per_s=round(w.total_tokens / ms * 1e3, 1),
               frac_of_bf16_peak=round(fl / ms / 1e9 / peaks["bf16_tflops"], 4),
               work_tflops=round((fl + 2.0 * w.dp * w.hkv * c["causal"]) / ms / 1e9, 3),
               kernels_ms={models[k]["name"]: round(v, 3) for k, v in kern_ms.items()},
               calls_ms={k: round(v, 3) for k, v in calls.items()},
               gpu_launches=int(launches), clocks=clk)
    del step
    torch.cuda.empty_cache()
    rec["device_peak_gb"] = round(torch.cuda.max_memory_allocated() / 1e9, 1)
    if args.dense:
        long = w.total_tokens > 200000
        rec["dense_sdpa"] = dense_sdpa(w, inp, steps=dense_steps, warmup=1,
                                       warm_tokens=8192 if long else None)
    if args.cpu_baseline and cpu_rows is not None:
        rec["cpu_baseline"] = cpu_baseline(w, inp, cpu_rows, w.seed)
    del inp
    torch.cuda.empty_cache()
    return rec


def run_select_only(args):
    """The selection call alone on the workload's inputs, for profiling: only
    cu_seqlens, q_p, k_p, the selection outputs and the selection workspace
    stay on the device.  Prints one JSON line with the call's time."""
    import block_sparse_attention_proxy_gb300 as m
    from block_sparse_attention_proxy_gb300.step import params_for

    dist_setup()
    m.load()
    w = synth.workload(args.workload)
    inp = make_device_inputs(w)
    cu, qp, kp = inp["cu_seqlens"], inp["q_p"], inp["k_p"]
    del inp
    torch.cuda.empty_cache()
    prm = params_for(cu.tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k)
    T, hkv, K = w.total_tokens, w.hkv, w.top_k
    out = dict(sel_idx=torch.empty(T, hkv, K, dtype=torch.int32, device="cuda"),
               sel_score=torch.empty(T, hkv, K, dtype=torch.float32, device="cuda"),
               sel_arg=torch.empty(T, hkv, K, dtype=torch.uint8, device="cuda"),
               plse=torch.empty(T, hkv, dtype=torch.float32, device="cuda"),
               tie=torch.empty(T, hkv, dtype=torch.uint8, device="cuda"))
    ws = m.workspace(m.msa_select_workspace_size(prm))

    def call():
        m.msa_proxy_select(prm, cu, qp, kp, out["sel_idx"], out["sel_score"], out["sel_arg"],
                           out["plse"], out["tie"], ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    if m.msa_get_device_status() != 0:
        raise RuntimeError(f"device status {m.msa_last_status_word():#x}")
    print(json.dumps(dict(workload=w.name, call="msa_proxy_select", steps=args.steps,
                          ms_per_call=round(e0.elapsed_time(e1) / max(1, args.steps), 3),
                          device_peak_gb=round(torch.cuda.max_memory_allocated() / 1e9, 2))),
          flush=True)


def run_ours(args):
    import block_sparse_attention_proxy_gb300 as m
    from block_sparse_attention_proxy_gb300.step import MSAStep, params_for

    world, rank, local = dist_setup()
    m.load()
    peaks = load_peaks()
    wanted = [n for n in args.configs.split(",") if n] if rank == 0 else []
    for n in wanted:
        if n not in PER_CONFIG:
            raise SystemExit(f"--configs: unknown workload {n!r} (choose from {', '.join(PER_CONFIG)})")
    configs = [n for n in PER_CONFIG if n in wanted and n != args.workload]
    # the CPU oracle on every row of the small workloads runs in a spawned
    # process while this one drives the GPU, started after the headline's
    # device and end-to-end timings (busy host cores slowed the host-link
    # copies of the end-to-end steps); the sampled-row baselines of this
    # process run after it has finished, so the two never share the cores
    oracle_proc, oracle_q = None, None
    full_rows = [n for n in configs if PER_CONFIG[n][3] is None]

    def start_oracle():
        nonlocal oracle_proc, oracle_q
        if args.cpu_baseline and full_rows:
            import multiprocessing as mp

            ctx = mp.get_context("spawn")
            oracle_q = ctx.Queue()
            oracle_proc = ctx.Process(target=_oracle_all_rows,
                                      args=(full_rows, max(1, (os.cpu_count() or 2) - 2), oracle_q),
                                      daemon=True)
            oracle_proc.start()

    w = synth.workload(args.workload)
    c = work_counts(w)
    inp = make_device_inputs(w)
    prm = params_for(inp["cu_seqlens"].tolist(), w.hq, w.hkv, w.d, w.dp, w.top_k)
    step = MSAStep(prm)
    K, W = args.steps, args.warmup
    ms_local, kern_ms, calls, launches, clk = time_steps(step, inp, K, W, world)
    ms = max_over_ranks(ms_local, world)
    fl = flops_effective(w, c)
    value = fl * world / ms / 1e9
    models = kernel_models(w, c)
    top = max(kern_ms, key=lambda k: kern_ms[k])
    mdl = models[top]
    if mdl["bound"] == "tensor":
        achieved = mdl["work"] / kern_ms[top] / 1e9
        peak = peaks["bf16_tflops"]
    else:
        achieved = mdl["work"] / kern_ms[top] / 1e6
        peak = peaks["hbm_gbs"]
    traffic = recorded_traffic(mdl["name"], w.name)
    roofline = dict(kernel=mdl["name"], bound=mdl["bound"], achieved=round(achieved, 2),
                    peak=peak, unit=mdl["unit"], frac=round(achieved / peak, 4),
                    traffic=traffic, peak_source=f"{peaks['source']} (MEASURED_PEAKS.json)"
                    if peaks["source"] == "measured" else "fallback",
                    kernel_ms=round(kern_ms[top], 3), algorithmic_per_launch=mdl["work"])
    per_kernel = {models[k]["name"]: dict(ms=round(kern_ms[k], 3), bound=models[k]["bound"],
                                          achieved=round(models[k]["work"] / kern_ms[k] /
                                                         (1e9 if models[k]["bound"] == "tensor"
                                                          else 1e6), 2),
                                          unit=models[k]["unit"]) for k in kern_ms}
    device_peak = round(torch.cuda.max_memory_allocated() / 1e9, 1)

    # ---- end to end through the C ABI with host buffers ----
    e2e = run_e2e(w, inp, step, fl, K, W, world) if args.e2e else None
    start_oracle()
    del step
    torch.cuda.empty_cache()
    dense = dense_sdpa(w, inp) if (args.dense and rank == 0) else None

    # ---- the other workloads of the metric's range ----
    per_config = {}
    for name in configs:
        Kc, Wc, dsteps, rows = PER_CONFIG[name]
        try:
            per_config[name] = measure_config(name, peaks, args, None, dsteps, Kc, Wc)
        except torch.cuda.OutOfMemoryError as ex:
            per_config[name] = dict(unavailable=f"out of device memory: {str(ex)[:160]}")
            torch.cuda.empty_cache()
    cpu = None
    if oracle_proc is not None:
        oracle_proc.join()
        while not oracle_q.empty():
            name, rec = oracle_q.get()
            per_config[name]["cpu_baseline"] = rec
    if args.cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(w, inp, args.cpu_rows, w.seed)
        for name in configs:
            rows = PER_CONFIG[name][3]
            if rows is not None and "unavailable" not in per_config[name]:
                wc = synth.workload(name)
                ic = make_device_inputs(wc)
                per_config[name]["cpu_baseline"] = cpu_baseline(wc, ic, rows, wc.seed)
                del ic
                torch.cuda.empty_cache()
    if configs:
        per_config[w.name] = dict(workload=config_of(w)["workload"], tokens=w.total_tokens,
                                  steps=K, warmup=W, ms_per_step=round(ms, 3),
                                  tflops=round(value / world, 3),
                                  tokens_per_s=round(w.total_tokens / ms * 1e3, 1),
                                  frac_of_bf16_peak=round(value / world / peaks["bf16_tflops"], 4),
                                  kernels_ms={k: v["ms"] for k, v in per_kernel.items()},
                                  calls_ms={k: round(v, 3) for k, v in calls.items()},
                                  device_peak_gb=device_peak, dense_sdpa=dense,
                                  cpu_baseline=cpu, note="the headline line's own measurement")

    line = dict(
        metric=METRIC, value=round(value, 3), unit=UNIT, n_gpus=world, steps=K, warmup=W,
        ms_per_step=round(ms, 3), higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="bf16", data="synthetic (seeded; see synth/)",
        config=config_of(w, world),
        tokens_per_s=round(w.total_tokens * world / ms * 1e3, 1),
        work_tflops=round((fl + 2.0 * w.dp * w.hkv * c["causal"]) * world / ms / 1e9, 3),
        frac_of_bf16_peak=round(value / world / peaks["bf16_tflops"], 4),
        frac_of_bf16_sustained=round(value / world / peaks["bf16_tflops_sustained"], 4),
        device_peak_gb=device_peak,
        roofline=roofline, kernels=per_kernel,
        calls_ms={k: round(v, 3) for k, v in calls.items()},
        cpu_baseline=cpu, e2e=e2e, gpu_launches=int(launches), clocks=clk,
        dense_sdpa=dense, per_config=per_config or None,
    )
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


E2E_DEPTH = 3


def run_e2e(w, inp, step, fl, K, W, world) -> dict:
    """The same metric end to end through the library's host-input API
    (HostInputStep): every step copies its inputs from pinned host memory to
    the device and its results (O, LSE, the five gradients and the loss) back
    to pinned host memory, all inside the timed region.  The copies run on two
    copy streams and overlap the kernels (inputs of later calls and of the next
    steps; O during the backward; the gradients during the next steps).  Three
    input and output sets rotate (E2E_DEPTH), so a copy that runs slow for a
    while (host-link copy rates vary from step to step) holds the kernels back
    only once it is two steps behind."""
    from block_sparse_attention_proxy_gb300.step import HostInputStep

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    names_in = ("q", "k", "v", "q_p", "k_p", "dO", "cu_seqlens")
    host_in = {n: inp[n].to("cpu").pin_memory() for n in names_in}
    hs = HostInputStep(step.params, inp, step=step, depth=E2E_DEPTH)
    host_out = hs.allocate_host_outputs()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    def e2e_step():
        hs(host_in, host_out=host_out)

    for _ in range(max(1, W)):
        e2e_step()
    hs.wait_outputs()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = E(), E()
    e0.record()
    hs.copy_stream.wait_event(e0)  # no copy of the timed steps starts before e0
    hs.out_stream.wait_event(e0)
    for _ in range(K):
        e2e_step()
    hs.wait_outputs()  # the last step's results are on the host before e1
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / K, world)
    # copy rates alone (one step's inputs / results, nothing else running), for
    # reading the number above: the copies hide behind the kernels while they
    # take less than a step
    c0, c1, c2, c3 = E(), E(), E(), E()
    c0.record(hs.copy_stream)
    with torch.cuda.stream(hs.copy_stream):
        for n in names_in:
            hs.bufs[0][n].copy_(host_in[n], non_blocking=True)
    c1.record(hs.copy_stream)
    torch.cuda.synchronize()
    c2.record(hs.out_stream)
    with torch.cuda.stream(hs.out_stream):
        for n, t in host_out.items():
            t.copy_(step.out[n], non_blocking=True)
    c3.record(hs.out_stream)
    torch.cuda.synchronize()
    return dict(value=round(fl * world / ms_e2e / 1e9, 3), unit=UNIT,
                ms_per_step=round(ms_e2e, 3), h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                tokens_per_s=round(w.total_tokens * world / ms_e2e * 1e3, 1),
                returned=list(host_out), buffer_sets=E2E_DEPTH,
                h2d_gb_per_s_alone=round(h2d / (c0.elapsed_time(c1) * 1e6), 1),
                d2h_gb_per_s_alone=round(d2h / (c2.elapsed_time(c3) * 1e6), 1))


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    from oracle import OracleParams, row_reference

    w = synth.workload(args.workload)
    inp = synth.make_inputs(w, device="cpu")
    prm = OracleParams(w.hq, w.hkv, w.d, w.dp, w.top_k)
    cu = inp["cu_seqlens"].tolist()
    rows_per_step = args.ref_rows
    rng = np.random.default_rng(w.seed)

    def one_step():
        rows = rng.integers(0, w.total_tokens, size=rows_per_step)
        pairs = 0
        for t in rows:
            row_reference(inp, prm, int(t), contributions=True)
            a = max(x for x in cu[:-1] if x <= t)
            i = int(t) - a
            pairs += min(i // 128, w.top_k - 1) * 128 + i % 128 + 1
        return 14.0 * w.d * w.hq * pairs

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += one_step()
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    ms = dt / args.steps * 1e3
    sample = (f"each step: {rows_per_step} seeded query rows of the {w.name} workload (all heads "
              f"and groups, fwd+bwd incl. dK/dV/dk_p contributions)")
    line = dict(
        metric=METRIC, value=round(value, 6), unit=UNIT, n_gpus=int(os.environ.get("WORLD_SIZE", 1)),
        steps=args.steps, warmup=args.warmup, ms_per_step=round(ms, 3), higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype="f64", data="synthetic (seeded; see synth/)",
        config=config_of(w, world),
        impl="reference",
        cpu_baseline=dict(kind="oracle", cores=os.cpu_count(), sample=sample, value=round(value, 6),
                          unit=UNIT),
        e2e=dict(value=round(value, 6), unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
    )
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="128k", choices=synth.WORKLOADS)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-dense", dest="dense", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false",
                    help="skip the end-to-end leg (profiling runs only)")
    ap.add_argument("--configs", default=",".join(PER_CONFIG),
                    help="comma-separated workloads measured besides the headline one "
                         "(per_config records); default: the whole range")
    ap.add_argument("--no-configs", dest="configs", action="store_const", const="",
                    help="measure only the headline workload (no per_config records)")
    ap.add_argument("--only-select", action="store_true",
                    help="profiling: time the selection call alone (few GB on the device)")
    ap.add_argument("--cpu-rows", type=int, default=128)
    ap.add_argument("--ref-rows", type=int, default=4)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.only_select:
        run_select_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
