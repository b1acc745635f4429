#!/usr/bin/env python
"""Benchmark of the Gemma-4-assistant MTP drafter on GB300.

One step = one pass of the whole hot path on one batch: a draft block (n_draft drafter
steps: pre_projection, 4 Q-only blocks over the shared K, post_projection, centroid head
+ argmax) followed by greedy verification of the drafted tokens against synthetic target
logits. Workload: the E2B shape, B=1, ctx 4096, draft block 4 (seeded synthetic inputs).

Metric: draft tokens/s (= B * n_draft / step time) and us per drafter step, plus the
fraction of the HBM roofline reached by the persistent draft-block kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mtp|reference]

Multi-GPU: independent replicas, one process per GPU (torchrun); per-GPU work is fixed
("weak" scaling) and nothing is exchanged on the data path.
--impl reference times the CPU oracle (the reference arm of this build) on the host.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft tokens/s and µs per drafter step (E2B shape, B=1) + % HBM roofline"
UNIT = "draft tokens/s"
L2_FLUSH_BYTES = 256 << 20          # > 2x the 129 MB L2
HBM_FALLBACK_GBS = 6800.0


# ---------------------------------------------------------------------------------------
# workload and algorithmic bytes
# ---------------------------------------------------------------------------------------

SPARSE_HEAD = {"auto": 0, "per-sequence": 1, "cluster-major": 2}  # enum mtp_sparse_head


def workload(index: int):
    from mtp_synth import configs as C
    cfg = C.config(index)
    return cfg.shape, cfg.workload


def algorithmic_bytes_per_step(shape, B: int, ctx_lens) -> dict:
    """Unique bytes one drafter step must read, for the whole batch: every weight once
    (storage dtype; norm gains fp32), per sequence the shared-K range each attention type
    attends (once per type, not once per layer), the k*vsc gathered token_embd rows with
    their int32 ids, and the target-embedding row of the input token."""
    eb = 2 if shape.dtype == "bf16" else 4
    H, bb, F = shape.hidden, shape.backbone, shape.ffn
    w = H * 2 * bb + bb * H
    g = H
    for t in shape.layer_types:
        d = shape.head_dim(t)
        w += 2 * H * shape.n_head * d + 3 * H * F
        g += 4 * H + d
    if shape.use_ordered_embeddings:
        w += shape.n_centroids * H
    weights = w * eb + g * 4
    kv = rows = embed = 0
    for L in ctx_lens:
        L = int(L)
        if "F" in shape.layer_types:
            kv += L * shape.n_kv_head * shape.head_dim_full * eb
        if "S" in shape.layer_types:
            kv += min(L, shape.window) * shape.n_kv_head * shape.head_dim_swa * eb
        if shape.use_ordered_embeddings:
            n = shape.top_k * shape.vsc
            rows += n * H * eb + n * 4
        else:
            rows += 0
        embed += bb * eb
    if not shape.use_ordered_embeddings:
        weights += shape.vocab * H * eb     # dense tied head reads every row once per step
    total = weights + kv + rows + embed
    return dict(weights=weights, kv=kv, rows=rows, embed=embed, total=total)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback 6.8 TB/s"


# The device code each captured kernel is compiled from (its translation unit and the device
# headers it includes); other kernels hash the whole csrc directory.
KERNEL_SOURCES = {"k_block_c2": ("mtp_c2.cu", "mtp_c2.cuh", "mtp_common.cuh"),
                  "k_block_gr": ("mtp_grid.cu", "mtp_grid.cuh", "mtp_common.cuh")}


def kernel_source_hash(kernel: str = "") -> str:
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "mtp_speculative_decoding_gemma4_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel)
    paths = ([os.path.join(pkg, n) for n in names] if names else sorted(glob.glob(os.path.join(pkg, "*"))))
    for p in paths:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, config_index: int):
    """DRAM bytes per launch from a committed ncu capture of the same kernel source, else
    None (also None once the kernel source changed since the capture)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{kernel}@config{config_index}"]
        if e.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------------------
# replicas: one process per GPU, nothing exchanged on the data path
# ---------------------------------------------------------------------------------------

def max_over_ranks(values, dist, device="cuda"):
    """Each timing's maximum over the ranks (the slowest replica bounds the job); the values
    unchanged without a process group."""
    if not dist:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the draft tokens of every replica over the slowest step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


# ---------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------------------

def _to_dev(arr, dtype, torch):
    import numpy as np
    if dtype == "bf16" and arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def pct(values, q: float) -> float:
    """The q-quantile (0..1) of the values, nearest rank."""
    v = sorted(values)
    return v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]


def run_mtp(args, rank: int, world: int, dist):
    import numpy as np
    import torch

    import __graft_entry__ as ge
    ge.build()
    from mtp_speculative_decoding_gemma4_gb300 import Drafter, verify_greedy
    from mtp_synth import gen as G

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    shape, wl = workload(args.config)
    B, n = wl.batch, wl.n_draft
    w = G.make_weights(shape, wl.seed)
    inp = G.make_step_inputs(shape, wl, wl.seed)
    dt = shape.dtype
    wd = {k: (None if getattr(w, k) is None else _to_dev(getattr(w, k), "f32" if k == "out_norm" else
                                                        ("i32" if k == "token_ordering" else dt), torch))
          for k in ("pre_proj", "post_proj", "out_norm", "token_embd", "centroids", "token_ordering")}
    wd["layers"] = [{k: (v if k == "layer_scalar" else _to_dev(v, "f32" if k.endswith("norm") else dt, torch))
                     for k, v in L.items()} for L in w.layers]
    dr = Drafter(shape, wd, _to_dev(w.target_embed, dt, torch), max_batch=B, max_ctx=wl.ctx)
    dr.set_path(args.path)
    dr.set_sparse_head(SPARSE_HEAD[args.sparse_head])
    d = dict(hidden=_to_dev(inp.hidden, dt, torch), last_token=_to_dev(inp.last_token, "i32", torch),
             ctx_len=_to_dev(inp.ctx_len, "i32", torch), pos=_to_dev(inp.pos, "i32", torch),
             k_swa=None if inp.k_swa is None else _to_dev(inp.k_swa, dt, torch),
             k_full=None if inp.k_full is None else _to_dev(inp.k_full, dt, torch))
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    out_tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out_v = torch.empty((B, n + 1), dtype=torch.int32, device="cuda")

    def draft():
        dr.draft_block(d["hidden"], d["last_token"], d["k_swa"], d["k_full"], d["ctx_len"], d["pos"], n,
                       want_hidden=False, out_tokens=out_tok, stream=sh)

    # synthetic target logits with a planted maximum agreeing with the draft w.p. 0.6
    draft()
    torch.cuda.synchronize()
    agree, alt_raw = G.round_tables(B, n, shape.vocab, 0.6, wl.seed, 0)
    tgt = G.planted_targets(out_tok.cpu().numpy(), agree, alt_raw, shape.vocab)
    base = G.base_target_logits(B, n + 1, shape.vocab, wl.seed)
    base[np.arange(B)[:, None], np.arange(n + 1)[None, :], tgt] = G.bf16_bits(np.float32([G.PLANT_VALUE]))[0]
    logits = _to_dev(base, "bf16", torch)

    def verify():
        verify_greedy(logits, out_tok, accept_len=acc, out_tokens=out_v, stream=sh)

    if args.profile_blocks:
        # exactly this many steps (draft block + verify), nothing timed: the program named by
        # the ncu captures
        for _ in range(args.profile_blocks):
            draft()
            verify()
        torch.cuda.synchronize()
        assert dr.status() == 0
        return None

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(max(3, args.warmup)):
        draft(); verify()
    torch.cuda.synchronize()
    assert dr.status() == 0

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(K):
            flush.zero_()                      # evict the previous step's working set from L2
            ev[i][0].record(stream)
            draft()
            ev[i][1].record(stream)
            verify()
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    draft_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms_per_step = sum(step_ms) / K
    draft_ms_mean = sum(draft_ms) / K
    spread = {"step_ms_median": statistics.median(step_ms), "step_ms_p90": pct(step_ms, 0.9),
              "draft_ms_median": statistics.median(draft_ms), "draft_ms_p90": pct(draft_ms, 0.9)}
    assert dr.status() == 0

    # sampled verification (temperature 1, seeded uniforms) of the same drafts and logits
    from mtp_speculative_decoding_gemma4_gb300 import verify_sample
    gen = torch.Generator(device="cuda")
    gen.manual_seed(wl.seed)
    u_acc = torch.rand((B, n), device="cuda", generator=gen)
    u_smp = torch.rand((B, n + 1), device="cuda", generator=gen)
    acc_s = torch.empty(B, dtype=torch.int32, device="cuda")
    out_s = torch.empty((B, n + 1), dtype=torch.int32, device="cuda")
    vs_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        vs_ev[i][0].record(stream)
        verify_sample(logits, out_tok, 1.0, u_acc, u_smp, accept_len=acc_s, out_tokens=out_s, stream=sh)
        vs_ev[i][1].record(stream)
    torch.cuda.synchronize()
    vs_ms = sum(e[0].elapsed_time(e[1]) for e in vs_ev) / K
    vs_rows = int(torch.clamp(acc_s + 1, max=n + 1).sum().item())

    # warm-L2 reference figure: back-to-back steps, no flush
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        draft(); verify()
    e1.record(stream)
    torch.cuda.synchronize()
    warm_ms = e0.elapsed_time(e1) / K

    # end to end through the public API with host buffers: per step, H2D of the step's
    # inputs from pinned memory, the draft block and verify, D2H of the result, host wait
    # The step's inputs sit back to back (16-byte aligned) in one pinned host buffer and one
    # device buffer, so each step takes one H2D copy; the draft block reads views of the device
    # buffer. The results (verified tokens, accept lengths) share one device buffer, read back
    # by one D2H copy.
    ins = [d["hidden"], d["last_token"], d["pos"], d["ctx_len"]]
    offs, total = [], 0
    for t in ins:
        offs.append(total)
        total += (t.numel() * t.element_size() + 15) // 16 * 16
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    views = []
    for t, o in zip(ins, offs):
        nb = t.numel() * t.element_size()
        v = dev_in[o:o + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        host_in[o:o + nb].copy_(t.cpu().contiguous().view(torch.uint8).reshape(-1))
        views.append(v)
    d["hidden"], d["last_token"], d["pos"], d["ctx_len"] = views
    res = torch.empty(B * (n + 1) + B, dtype=torch.int32, device="cuda")
    out_v, acc = res[:B * (n + 1)].view(B, n + 1), res[B * (n + 1):]
    host_res = torch.empty_like(res, device="cpu").pin_memory()
    h2d = host_in.numel()
    d2h = host_res.numel() * 4
    e2e_s = []
    for i in range(K):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dev_in.copy_(host_in, non_blocking=True)
        draft(); verify()
        host_res.copy_(res, non_blocking=True)
        stream.synchronize()
        e2e_s.append(time.perf_counter() - t0)
    e2e_step = sum(e2e_s) / K
    assert torch.equal(host_res[:B * (n + 1)].view(B, n + 1), out_v.cpu()), "e2e result read back"

    ms_per_step, e2e_step, draft_ms_mean, warm_ms = max_over_ranks([ms_per_step, e2e_step, draft_ms_mean, warm_ms],
                                                                    dist)

    if rank != 0:
        return None
    alg = algorithmic_bytes_per_step(shape, B, inp.ctx_len)
    per_launch = alg["total"] * n
    peak, peak_src = measured_peaks()
    achieved = per_launch / (draft_ms_mean * 1e-3) / 1e9
    tokens = B * n * world  # every replica drafts B * n tokens per step
    head = (3 if shape.use_ordered_embeddings else 1)
    if args.path in (2, 6, 7):
        launches_per_step = 2
    elif args.path == 5:  # per step: staging + tcgen05 GEMM per projection, attention, combine, head
        # per block: Q staging + GEMM, attention, combine (stages O's operand), O GEMM, FFN
        # staging, and either [gate ; up] with the gated-GELU epilogue + down GEMM or gate, up,
        # down staging, down; post_projection takes the centroid GEMM along when both tile
        per_block = 8 if shape.ffn % 64 == 0 else 10
        stacked_head = shape.use_ordered_embeddings and shape.backbone % 128 == 0
        launches_per_step = 1 + n * (2 + per_block * shape.n_layers + 2 + head - stacked_head) + 1 + 1
    else:
        launches_per_step = 1 + n * (2 + 6 * shape.n_layers + 2) + 1 + 1
    kernel_name = {1: "phase kernels", 2: "k_block (persistent draft block, grid barriers)",
                   5: "k_tc_gemm + phase kernels (tcgen05 projections)",
                   6: "k_block_c2 (streamed-tile cluster draft block, tensor-core projections)",
                   7: "k_block_gr (grid draft block: split weights resident in shared memory, cluster + "
                      "global exchanges)"}[args.path]
    res = {
        "metric": METRIC, "value": job_tokens_per_s(B * n, world, ms_per_step), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "median_ms": spread["step_ms_median"], "p90_ms": spread["step_ms_p90"],
        "us_per_drafter_step": ms_per_step * 1e3 / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{shape.name} drafter step: B={B}, ctx {wl.ctx}, draft block {n}, then greedy "
                               f"verify of [{B},{n + 1},{shape.vocab}] bf16 target logits",
                   "batch": B, "ctx": wl.ctx, "n_draft": n, "storage": shape.dtype,
                   "sparse_head": args.sparse_head,
                   "l2": "flushed before every timed step (256 MiB write)", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(kernel_name.split()[0], args.config),
                     "kernel": kernel_name,
                     "alg_bytes_per_launch": per_launch, "alg_bytes_per_step": alg, "peak_source": peak_src,
                     "kernel_ms": draft_ms_mean, "kernel_ms_median": spread["draft_ms_median"],
                     "kernel_ms_p90": spread["draft_ms_p90"]},
        "e2e": {"value": tokens / e2e_step, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step * 1e3},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
        "warm_l2": {"ms_per_step": warm_ms, "value": tokens / (warm_ms * 1e-3)},
        "accept_len_mean": float(acc.float().mean().item()),
        "verify_sample": {"temperature": 1.0, "us": vs_ms * 1e3, "rows_read": vs_rows,
                          "accept_len_mean": float(acc_s.float().mean().item()),
                          "achieved_gbs": vs_rows * shape.vocab * 2 / (vs_ms * 1e-3) / 1e9,
                          "kernel": "k_verify_sample (one thread-block cluster per sequence)"},
    }
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args, shape, wl, w, inp, base, seconds=args.cpu_seconds)
    return res


# ---------------------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------------------

def blas_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_step_runner(shape, wl, w, inp, base):
    import oracle as O
    s, W = O.Shape.of(shape), O.decode_weights(w)

    def one():
        blk = O.draft_block(s, W, inp.hidden, inp.last_token, inp.k_swa, inp.k_full, inp.ctx_len, inp.pos,
                            wl.n_draft)
        O.verify_greedy(base, blk.tokens)
        return blk
    return one


def _time_oracle(one, seconds: float, max_steps: int = 10000):
    one()
    t0 = time.perf_counter()
    steps = 0
    while True:
        one()
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or steps >= max_steps:
            return steps, el


def cpu_baseline(args, shape, wl, w, inp, base, seconds: float):
    """The oracle timed on the host cores (BLAS on every core), and again with one BLAS
    thread; nproc stated beside both."""
    one = oracle_step_runner(shape, wl, w, inp, base)
    steps, el = _time_oracle(one, seconds)
    res = {"value": steps * wl.batch * wl.n_draft / el, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
           "nproc": os.cpu_count(),
           "sample": f"{steps} full steps (draft block of {wl.n_draft} + verify) of the same workload, "
                     f"{el:.1f} s, NumPy fp64"}
    # the same oracle with one BLAS thread: the reference arm in a child process whose BLAS
    # libraries start single-threaded (nothing here can change the thread count of a BLAS
    # that is already loaded)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", WORLD_SIZE="1", RANK="0")
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--config", str(args.config),
           "--steps", str(max(2, int(args.cpu_seconds / 2))), "--warmup", "1"]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        line = [x for x in r.stdout.splitlines() if x.startswith("{")][-1]
        d = json.loads(line)
        res["single_thread"] = {"value": d["value"], "unit": UNIT, "cores": 1,
                                "sample": f"{d['steps']} full steps, one BLAS thread (child process)"}
    except Exception as e:
        res["single_thread"] = {"unavailable": f"single-thread oracle run failed: {type(e).__name__}"}
    return res


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return None
    import numpy as np
    from mtp_synth import gen as G
    shape, wl = workload(args.config)
    w = G.make_weights(shape, wl.seed)
    inp = G.make_step_inputs(shape, wl, wl.seed)
    B, n = wl.batch, wl.n_draft
    base = G.base_target_logits(B, n + 1, shape.vocab, wl.seed)
    one = oracle_step_runner(shape, wl, w, inp, base)
    blk = one()
    agree, alt_raw = G.round_tables(B, n, shape.vocab, 0.6, wl.seed, 0)
    tgt = G.planted_targets(blk.tokens, agree, alt_raw, shape.vocab)
    base[np.arange(B)[:, None], np.arange(n + 1)[None, :], tgt] = G.bf16_bits(np.float32([G.PLANT_VALUE]))[0]
    for _ in range(args.warmup):
        one()
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        t.append(time.perf_counter() - t0)
    ms = 1e3 * sum(t) / len(t)
    value = B * n / (ms * 1e-3)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "us_per_drafter_step": ms * 1e3 / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{shape.name} drafter step: B={B}, ctx {wl.ctx}, draft block {n}, then greedy "
                                   f"verify of [{B},{n + 1},{shape.vocab}] bf16 target logits",
                       "batch": B, "ctx": wl.ctx, "n_draft": n, "storage": shape.dtype,
                       "sparse_head": args.sparse_head,
                       "l2": "host run (the GPU arm flushes 256 MiB of L2 before every timed step)",
                       "parallelism": "host"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": f"{args.steps} full steps of the workload, NumPy fp64"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mtp", "reference"], default="mtp")
    ap.add_argument("--config", type=int, default=1, help="benchmark configuration index (default 1: E2B, B=1)")
    ap.add_argument("--path", type=int, default=-1,
                    help="1: one launch per phase, 2: persistent kernel with grid barriers, 5: phase kernels "
                         "with tcgen05 projections, 6: streamed-tile cluster kernel (one sequence), 7: grid "
                         "kernel (one sequence); default: 7 for B=1, else 5")
    ap.add_argument("--profile-blocks", type=int, default=0,
                    help="run exactly this many steps (draft block + verify) of the chosen path and exit without timing "
                         "(the program the ncu captures in profiles/ name)")
    ap.add_argument("--sparse-head", choices=sorted(SPARSE_HEAD), default="auto",
                    help="traversal of the centroid head's candidate rows in the batched paths: per sequence, "
                         "cluster-major (each selected cluster streamed once per step), or auto (per sequence)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.path < 0:
        bsz = workload(args.config)[1].batch
        args.path = 7 if bsz == 1 else 5

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1 and args.impl == "mtp":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group(backend="nccl")
        dist = tdist
    res = run_reference(args, rank, world) if args.impl == "reference" else run_mtp(args, rank, world, dist)
    if res is not None:
        print(json.dumps(res), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
