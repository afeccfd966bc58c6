"""Benchmark of one DFlash drafting step on GB300.

A step is the whole hot path for every request of the workload: inject the
S new tokens' target features into every drafter layer's paged KV cache,
draft one S-token block (one forward of the drafter), select the path, and
verify greedily against synthetic target tokens (S = 16 unless the workload
sets a smaller runtime block size).

Default workload (the JSON line's headline): the 27B-class drafter (5 layers,
hidden 5120, 40 q / 8 kv heads, FFN 17408, vocab 151936), 64 requests with
ragged contexts uniform in [16384, 32768] tokens in 64-token KV pages - the
largest configuration that fits one GPU, where the step is bound by streaming
~32 GB of draft KV.  In the same run (N = 1) the Qwen3-8B-shaped workloads
C1 (batch 1, context 2048), C2 (32 ragged requests, 1k-8k) and C3 (DFlash-2,
8 x 4096) are measured the same way and reported under "other_workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload C4|C1|C2|C3|C1S5|C2S5|C1F8|...] [--extra C1,C2,C3|none]
                  [--mode greedy|sampling]

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on the same workload instead (the deliberately slow reference arm).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import WORKLOADS, gen  # noqa: E402

METRIC = "drafted blocks/sec (16-tok) at batch×ctx on 1 GB300; attention HBM GB/s"
DEFAULT_WORKLOAD = "C4"
DEFAULT_EXTRA = "C1,C2,C3"
# GEMMs with at least this many token rows are measured against the tensor
# peak (ridge point of the measured bf16 rate over the measured HBM rate)
TENSOR_BOUND_TOKENS = 300
GEMM_NAMES = ("fc", "kv_inject", "qkv", "o_proj", "gate_up", "down", "lm_head", "lm_head_topk", "conv_coef")
# kernel source files whose ncu DRAM counters in profiles/traffic.json stay
# valid only while these files are unchanged
KERNEL_SOURCES = {"attention": ("attention.cu", "common.cuh"), "gemm": ("gemm_tc.cu", "common.cuh"),
                  "topk16": ("topk.cu",)}


def metric(cfg) -> str:
    return METRIC if cfg.block == 16 else METRIC.replace("(16-tok)", f"({cfg.block}-tok)")


FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def weight_bytes(cfg) -> float:
    """Bytes of GEMM weights one drafting step streams (every projection once)."""
    H, d, F, V = cfg.hidden, cfg.head_dim, cfg.ffn, cfg.vocab
    per_layer = (cfg.n_q_heads + 2 * cfg.n_kv_heads) * d * H + cfg.n_q_heads * d * H + 3 * F * H
    if cfg.use_conv:
        per_layer += 4 * (H // 8) * H
    n = cfg.n_layers * per_layer + V * H + H * cfg.feat_in
    return n * (1.0 if cfg.weight_fp8 else 2.0)


def kv_bytes_per_token(cfg) -> int:
    """Bytes of K and V one context token holds over all drafter layers (the
    block attention reads each once per step): 20 480 at 5 layers x 8 kv
    heads x 128 x bf16."""
    return cfg.n_layers * cfg.n_kv_heads * cfg.head_dim * 2 * (4 if cfg.dtype == "f32" else 2)


def attention_bytes_per_step(cfg, ctx) -> float:
    """Algorithmic bytes of the block attention in one step: every request's
    context plus the S tokens the step injected, plus the S block keys and
    values."""
    S = cfg.block
    return float(sum(int(c) + 2 * S for c in ctx)) * kv_bytes_per_token(cfg)


def prefill_injection_flops(cfg, tokens: int) -> float:
    """Dense flops of injecting `tokens` context tokens: the context-feature
    projection [tokens, n_sel*H_t] x [n_sel*H_t, H] and every layer's K and V
    projections [tokens, H] x [H, 2*nkv*d]."""
    return 2.0 * tokens * cfg.hidden * (cfg.feat_in + cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim)


def sample_requests(batch: int) -> list:
    """The requests the CPU oracle times: first, middle and last."""
    return sorted({0, batch // 2, batch - 1})


def workload_desc(wl):
    c = wl.cfg
    return (f"{wl.name}: {c.name} drafter (L={c.n_layers}, H={c.hidden}, {c.n_q_heads}q/{c.n_kv_heads}kv x "
            f"{c.head_dim}, F={c.ffn}, V={c.vocab}), batch {wl.batch}, context "
            f"{wl.ctx_lo if wl.ctx_lo == wl.ctx_hi else f'U[{wl.ctx_lo},{wl.ctx_hi}]'}, "
            f"{c.n_target_layers}x{c.target_hidden} target features, block size {c.block}, "
            f"{c.block} new tokens injected per step" + (", FP8 E4M3 weights (per-row scales)" if c.weight_fp8 else ""))


def source_sha16(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "block_diffusion_drafter_context_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when none exists or the kernel's source
    has changed since the counters were taken."""
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(tfile)).get(workload, {}).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("source_sha16") != source_sha16(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling during the timed region (clocks + throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []          # (host arrival time, fields)
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.perf_counter() + 3.0   # running before the timed region starts
            while not self.rows and time.perf_counter() < deadline:
                time.sleep(0.005)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.perf_counter(), parts))

    def mark(self, start: bool):
        """Host time of the timed region's start / end."""
        if start:
            self.t0 = time.perf_counter()
        else:
            self.t1 = time.perf_counter()
            deadline = self.t1 + 0.2               # one sample after the region ends
            while time.perf_counter() < deadline and not any(t > self.t1 for t, _ in self.rows):
                time.sleep(0.005)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = self.rows
        if self.t0 is not None and self.t1 is not None:
            inside = [r for t, r in rows if self.t0 <= t <= self.t1]
            after = [r for t, r in rows if t > self.t1][:1]
            rows = inside + after
        else:
            rows = [r for _, r in rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- multi-rank helpers
def rank_requests(batch: int, world: int, rank: int) -> range:
    """Contiguous shard of a batch of independent requests for one rank."""
    lo = batch * rank // world
    hi = batch * (rank + 1) // world
    return range(lo, hi)


def max_over_ranks(ms: float, dist=None, device=None) -> float:
    """Slowest rank's time (the job's time): all-reduce MAX when distributed."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_blocks_per_s(world: int, batch_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's blocks over the slowest rank's time."""
    return world * batch_per_rank * steps / (max_ms * 1e-3)


# ---------------------------------------------------------------- CPU oracle
def oracle_setup(wl, W, ctx, X_prefill, cu, requests=None, templates=None, table=None):
    """The oracle's context KV of each request (None for requests not listed)."""
    import oracle as O
    kvs = [None] * wl.batch
    for b in (range(wl.batch) if requests is None else requests):
        n = int(ctx[b])
        if templates is not None:
            tk, tv, pmap = templates
            kvs[b] = [(O.f64(k), O.f64(v)) for k, v in gen.template_request_kv(wl.cfg, tk, tv, pmap, table[b], n)]
        else:
            kvs[b] = O.inject_context(wl.cfg, W, X_prefill[cu[b]:cu[b + 1]], np.arange(n))
    return kvs


def oracle_step(wl, W, kvs, ctx, Xn, anchor, target, requests):
    import oracle as O
    outs = []
    S = wl.cfg.block
    for b in requests:
        outs.append(O.drafting_step(wl.cfg, W, kvs[b], int(ctx[b]), Xn[S * b:S * (b + 1)], int(anchor[b]),
                                    target[b]))
    return outs


def blas_threads() -> int:
    """Threads the oracle's BLAS runs on (what the CPU baseline used)."""
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(k)
        if v and v.isdigit():
            return int(v)
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_request_rate(wl, W, ctx, Xp, cu, Xn, anchor, target, templates, table, requests):
    """Oracle blocks/s on the listed requests (one full request-step each:
    inject S tokens, forward, top-16, select, verify), their KV set-up
    untimed; (blocks/s, seconds)."""
    kvs = oracle_setup(wl, W, ctx, Xp, cu, requests=requests, templates=templates, table=table)
    t0 = time.perf_counter()
    oracle_step(wl, W, kvs, ctx, Xn, anchor, target, requests)
    el = time.perf_counter() - t0
    return len(requests) / el, el


def oracle_probe(name: str) -> dict:
    """One request-step of the oracle on request 0 of `name` (run in a child
    process whose BLAS is limited to one thread)."""
    # the drawn cache state: the timed request-step is the same work, and the
    # single-threaded oracle would otherwise spend minutes on the prefill
    wl = dataclasses.replace(WORKLOADS[name], kv_fill="template")
    W, ctx, table, npages, cu, Xp, Xn, anchor = make_inputs(wl, prefill_requests=[0])
    tgt = np.zeros((wl.batch, wl.cfg.block), np.int32)
    v, el = oracle_request_rate(wl, W, ctx, Xp, cu, Xn, anchor, tgt, kv_templates(wl, npages), table, [0])
    return {"workload": name, "blocks_per_s": v, "seconds": el, "threads": blas_threads()}


def single_thread_oracle(names=("C0", "C1"), timeout=300) -> dict:
    """The oracle's request-step on one host thread, per workload."""
    out = {}
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for n in names:
        try:
            r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-probe", n],
                               capture_output=True, text=True, timeout=timeout, env=env, cwd=ROOT)
            line = [l for l in r.stdout.splitlines() if l.startswith("{")]
            out[n] = json.loads(line[-1]) if (r.returncode == 0 and line) else {"error": r.stderr[-300:]}
        except Exception as e:
            out[n] = {"error": f"{type(e).__name__}: {e}"}
    return out


# ---------------------------------------------------------------- inputs
def make_inputs(wl, prefill_requests=None):
    """Seeded inputs of a workload.  The context prefill's target features
    (when the workload injects its context) are generated for the listed
    requests only (all when None); other requests' rows are left empty."""
    cfg = wl.cfg
    W = gen.make_weights(cfg, wl.seed)
    ctx = gen.context_lengths(wl)
    B = len(ctx)
    table, npages = gen.page_table(ctx + cfg.block, cfg.page_size, wl.seed)
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    Xp = None
    if wl.kv_fill != "template":
        if prefill_requests is None:
            Xp = gen.target_hidden(cfg, int(ctx.sum()), wl.seed, "prefill")
        else:
            # the same values as the whole prefill at the listed requests' rows
            hi = max(int(cu[b + 1]) for b in prefill_requests)
            Xp = gen.target_hidden(cfg, hi, wl.seed, "prefill")
    Xn = gen.target_hidden(cfg, cfg.block * B, wl.seed, "step")
    anchor = gen.anchors(wl)
    return W, ctx, table, npages, cu, Xp, Xn, anchor


def kv_templates(wl, npages):
    """(K templates, V templates, page map) of a drawn cache state, else None."""
    if wl.kv_fill != "template":
        return None
    tk, tv = gen.kv_templates(wl.cfg, wl.kv_templates, wl.seed)
    return tk, tv, gen.kv_page_map(wl.cfg, npages, wl.kv_templates, wl.seed)


def bench_workload(name: str, layers=None, batch=None, ctx=None, vocab=None) -> "Workload":
    """The workload as the bench runs it.  Contexts whose prefill features
    would take minutes to generate on the host (C2: ~150 k tokens x 20 480
    features) start from a drawn cache state instead; the timed step is the
    same work either way.  layers / batch / ctx (lo, hi) / vocab shrink a
    workload for small profiling cases (the name then says so)."""
    wl = WORKLOADS[name]
    cfg_kw = {k: v for k, v in (("n_layers", layers), ("vocab", vocab)) if v}
    wl_kw = {}
    if batch:
        wl_kw["batch"] = batch
    if ctx:
        wl_kw["ctx_lo"], wl_kw["ctx_hi"] = ctx
    if cfg_kw or wl_kw:
        tag = ",".join(f"{k}={v}" for k, v in list(cfg_kw.items()) + list(wl_kw.items()))
        wl = dataclasses.replace(wl, name=f"{wl.name}[{tag}]", cfg=dataclasses.replace(wl.cfg, **cfg_kw), **wl_kw)
    if wl.kv_fill != "template" and wl.batch * wl.ctx_hi > 100_000:
        wl = dataclasses.replace(wl, kv_fill="template")
    return wl


def run_reference(args, wl):
    """The reference arm: the fp64 oracle on the host cores.  Each step is a
    bounded sample of the workload: one request's full drafting step,
    cycling through the first, middle and last request; blocks/s is one
    block per request-step (every request is independent of the others)."""
    reqs = sample_requests(wl.batch)
    W, ctx, table, npages, cu, Xp, Xn, anchor = make_inputs(wl, prefill_requests=reqs)
    t0 = time.time()
    kvs = oracle_setup(wl, W, ctx, Xp, cu, requests=reqs, templates=kv_templates(wl, npages), table=table)
    setup_s = time.time() - t0
    zeros = np.zeros((wl.batch, wl.cfg.block), np.int32)
    first = oracle_step(wl, W, kvs, ctx, Xn, anchor, zeros, reqs)
    draft = np.zeros((wl.batch, wl.cfg.block - 1), np.int32)
    for b, o in zip(reqs, first):
        draft[b] = o["draft"]
    target = gen.target_ids(draft, wl.p_accept, wl.cfg.vocab, seed=wl.seed)
    for i in range(args.warmup):
        oracle_step(wl, W, kvs, ctx, Xn, anchor, target, [reqs[i % len(reqs)]])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(wl, W, kvs, ctx, Xn, anchor, target, [reqs[i % len(reqs)]])
    el = time.perf_counter() - t0
    v = args.steps / el
    cores = blas_threads()
    line = {"impl": "reference", "metric": metric(wl.cfg), "value": v, "unit": "blocks/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(wl), "batch": wl.batch,
                                            "ctx": int(ctx.max())},
            "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": cores, "nproc": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"each step is one request's full drafting step (inject {wl.cfg.block} "
                                       f"tokens, forward, top-16, select, verify), cycling through requests "
                                       f"{reqs} of {wl.batch}; blocks/s = request-steps/s, extrapolated "
                                       f"linearly to the batch (requests are independent); oracle KV set-up "
                                       f"({setup_s:.1f} s) untimed"},
            "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def run_workload(args, wl, steps, warmup, world, local, dev, headline):
    """Set up `wl` on the GPU, time the step and return its measurements."""
    import torch
    import torch.distributed as dist
    from block_diffusion_drafter_context_gb300 import binding as Bd
    from block_diffusion_drafter_context_gb300.drafter import Drafter, PagedKV, to_device

    cfg = wl.cfg
    t_setup = time.time()
    cpu_reqs = sample_requests(wl.batch) if headline else [0]
    W, ctx, table, npages, cu, Xp, Xn, anchor = make_inputs(wl)
    B, S, J = wl.batch, cfg.block, cfg.block - 1
    prefill = 0 if wl.kv_fill == "template" else int(ctx.max())
    dr = Drafter(cfg, W, max_batch=B, max_new_tokens=max(S * B, prefill), device=dev)
    Bd.dflash_set_gemm_pairs(dr.ctx, bool(args.gemm_pairs))
    Bd.dflash_set_fused_topk(dr.ctx, bool(args.fused_topk))
    kv = PagedKV(cfg, table, npages, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    templates = kv_templates(wl, npages)
    if templates is not None:
        # drawn cache state: template pages mapped onto the pool
        kv.fill_from_templates(*templates)
    else:
        # prefill: inject the whole context, one request at a time through a
        # view of its page-table row
        ctx0 = torch.zeros(B, dtype=torch.int32, device=dev)
        ctx_n = torch.empty(B, dtype=torch.int32, device=dev)
        for b in range(B):
            one_cu = to_device(np.array([0, ctx[b]], np.int32), dev)
            Bd.dflash_inject_context(dr.ctx, kv.row(b), to_device(Xp[cu[b]:cu[b + 1]], dev), one_cu,
                                     int(ctx[b]), ctx0[:1], ctx_n[b:b + 1], 1, dr.workspace, dr.ws_bytes, stream)
    torch.cuda.synchronize()
    n_b = to_device(ctx.astype(np.int32), dev)
    cu_new = to_device((S * np.arange(B + 1)).astype(np.int32), dev)
    Xn_d = to_device(Xn, dev)
    anc_d = to_device(anchor, dev)
    ctx_after = torch.empty(B, dtype=torch.int32, device=dev)
    topk_ids = torch.empty((B, J, 16), dtype=torch.int32, device=dev)
    topk_logits = torch.empty((B, J, 16), dtype=torch.float32, device=dev)
    hfin = torch.empty((B, S, cfg.hidden), dtype=dr.act_dtype, device=dev)
    draft = torch.empty((B, J), dtype=torch.int32, device=dev)
    scores = torch.empty((B, J, 16, 16), dtype=torch.float32, device=dev) if cfg.use_selector else None
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    bonus = torch.empty(B, dtype=torch.int32, device=dev)
    com = torch.empty((B, S), dtype=torch.int32, device=dev)
    target_d = torch.zeros((B, S), dtype=torch.int32, device=dev)
    sampling = args.mode == "sampling"
    if sampling:
        # sampling mode: draft drawn over the path scores (T = 1) and rejection
        # verification against target logits resident in HBM (in serving they
        # come from the target model on the same GPU); seeded uniforms
        rng = np.random.default_rng(wl.seed)
        uni = rng.random((B, J)).astype(np.float32)
        ua = rng.random((B, J)).astype(np.float32)
        ub = rng.random(B).astype(np.float32)
        uni_d, ua_d, ub_d = (torch.from_numpy(a).to(dev) for a in (uni, ua, ub))
        zt_d = torch.from_numpy(gen.normal((B, S, cfg.vocab), 1.5, wl.seed, "target_logits")).to(dev)
        probs = torch.empty((B, J, 16), dtype=torch.float32, device=dev)

    def step(x_in=Xn_d, a_in=anc_d, t_in=None):
        st = torch.cuda.current_stream().cuda_stream
        t_in = target_d if t_in is None else t_in
        Bd.dflash_inject_context(dr.ctx, kv.struct, x_in, cu_new, S * B, n_b, ctx_after, B, dr.workspace,
                                 dr.ws_bytes, st)
        Bd.dflash_draft_block(dr.ctx, kv.struct, ctx_after, a_in, B, topk_ids, topk_logits, hfin, None,
                              dr.workspace, dr.ws_bytes, st)
        if sampling:
            Bd.dflash_sample_path(dr.ctx, a_in, topk_ids, topk_logits, hfin, B, 1.0, uni_d, draft, probs, scores,
                                  dr.workspace, dr.ws_bytes, st)
            Bd.dflash_verify_rejection(dr.ctx, zt_d, draft, topk_ids, probs, ua_d, ub_d, B, acc, bonus, com,
                                       dr.workspace, dr.ws_bytes, st)
            return
        Bd.dflash_select_path(dr.ctx, a_in, topk_ids, topk_logits, hfin, B, draft, scores, dr.workspace,
                              dr.ws_bytes, st)
        Bd.dflash_verify_greedy(draft, t_in, B, S, acc, bonus, com, st)

    # synthetic target tokens from the step's own draft (identical every step)
    step()
    torch.cuda.synchronize()
    gpu_draft = draft.cpu().numpy()
    tgt = gen.target_ids(gpu_draft, wl.p_accept, cfg.vocab, seed=wl.seed)
    target_d.copy_(torch.from_numpy(tgt))
    setup_s = time.time() - t_setup

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert dr.status() == 0, "device status after warm-up"

    # the step's launches, captured once into a CUDA graph (no host work per launch)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()

    def timed(fn, k):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(k):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), dist if world > 1 else None, dev)
        if world > 1:
            dist.barrier()
        return ms

    clocks = None
    if headline:
        with ClockSampler(local) as cs:
            cs.mark(True)
            ms = timed(graph.replay, steps)
            cs.mark(False)
        clocks = cs.summary()
    else:
        ms = timed(graph.replay, steps)
    ms_eager = timed(step, steps)
    assert dr.status() == 0, "device status after the timed region"

    # ---- instrumented pass: CUDA events around every launch, captured with
    # the K steps into one graph so host gaps do not enter the durations
    Bd.dflash_profile_begin(dr.ctx)      # eager pass first: creates the event pool outside capture
    for _ in range(steps):
        step()
    Bd.dflash_profile_end(dr.ctx)
    Bd.dflash_profile_begin(dr.ctx)
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prof):
        for _ in range(steps):
            step()
    g_prof.replay()
    torch.cuda.synchronize()
    stats = Bd.dflash_profile_end(dr.ctx)
    launches = sum(s["launches"] for s in stats)
    del g_prof

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs from pinned host memory, runs the four C-ABI calls
    # (eagerly: host-side argument checks and launches inside the timed
    # region; or as the captured graph) and reads its result back
    pin_x = torch.from_numpy(Xn.view(np.int16) if Xn.dtype == np.uint16 else Xn).pin_memory()
    pin_a = torch.from_numpy(anchor).pin_memory()
    # per-step host inputs: the target's tokens (greedy) or the step's uniforms (sampling)
    pin_t = (torch.from_numpy(np.concatenate([uni.ravel(), ua.ravel(), ub])).pin_memory() if sampling
             else torch.from_numpy(tgt).pin_memory())
    uni_all = torch.cat([uni_d.view(-1), ua_d.view(-1), ub_d.view(-1)]) if sampling else None
    out_acc = torch.empty(B, dtype=torch.int32).pin_memory()
    out_bonus = torch.empty(B, dtype=torch.int32).pin_memory()
    out_com = torch.empty((B, S), dtype=torch.int32).pin_memory()
    x_dev = Xn_d.view(torch.int16) if Xn.dtype == np.uint16 else Xn_d
    cur = torch.cuda.current_stream()

    def e2e(run):
        def one():
            x_dev.copy_(pin_x, non_blocking=True)
            anc_d.copy_(pin_a, non_blocking=True)
            if sampling:
                uni_all.copy_(pin_t, non_blocking=True)
                uni_d.view(-1).copy_(uni_all[:B * J], non_blocking=True)
                ua_d.view(-1).copy_(uni_all[B * J:B * 2 * J], non_blocking=True)
                ub_d.copy_(uni_all[B * 2 * J:], non_blocking=True)
            else:
                target_d.copy_(pin_t, non_blocking=True)
            run()
            out_acc.copy_(acc, non_blocking=True)
            out_bonus.copy_(bonus, non_blocking=True)
            out_com.copy_(com, non_blocking=True)
            cur.synchronize()   # the host reads the step's result before the next step
        return one

    e2e_eager, e2e_graph = e2e(step), e2e(graph.replay)
    for _ in range(2):
        e2e_eager()
        e2e_graph()
    ms_e2e = timed(e2e_eager, steps)
    ms_e2e_graph = timed(e2e_graph, steps)
    h2d = pin_x.numel() * pin_x.element_size() + pin_a.numel() * 4 + pin_t.numel() * 4
    d2h = (out_acc.numel() + out_bonus.numel() + out_com.numel()) * 4
    assert dr.status() == 0, "device status after the end-to-end passes"
    gpu_acc = out_acc.numpy().copy()
    del graph

    # ---- prefill injection: request 0's whole context injected again into
    # its own slots (the same values): the large-M context-feature and K/V
    # projection GEMMs, measured apart from the step
    prefill_inj = None
    if Xp is not None and world == 1:
        try:
            T0 = int(ctx[0])
            x0 = to_device(Xp[cu[0]:cu[1]], dev)
            cu0 = to_device(np.array([0, T0], np.int32), dev)
            c_in = torch.zeros(1, dtype=torch.int32, device=dev)
            c_out = torch.empty(1, dtype=torch.int32, device=dev)
            row0 = kv.row(0)

            def inject_all():
                Bd.dflash_inject_context(dr.ctx, row0, x0, cu0, T0, c_in, c_out, 1, dr.workspace, dr.ws_bytes,
                                         torch.cuda.current_stream().cuda_stream)

            for _ in range(3):
                inject_all()
            reps = 5
            ms_inj = timed(inject_all, reps) / reps
            Bd.dflash_profile_begin(dr.ctx)
            inject_all()
            st_inj = Bd.dflash_profile_end(dr.ctx)
            assert dr.status() == 0, "device status after the prefill injection"
            g_inj = sum(s["ms"] for s in st_inj if s["name"] in ("fc", "kv_inject"))
            fl = prefill_injection_flops(cfg, T0)
            pk_i, src_i = peaks()
            tf = fl / (g_inj * 1e-3) / 1e12 if g_inj > 0 else None
            prefill_inj = {"tokens": T0, "ms": ms_inj, "gemm_ms": g_inj, "gemm_flops": fl, "gemm_tflops": tf,
                           "peak_tflops": float(pk_i["bf16_tflops"]), "peak_source": f"{src_i} bf16_tflops (burst)",
                           "frac": tf / float(pk_i["bf16_tflops"]) if tf else None,
                           "launches": sum(s["launches"] for s in st_inj)}
        except Exception as e:   # reported, never fatal to the step's line
            prefill_inj = {"error": f"{type(e).__name__}: {e}"}

    dr.close()
    del dr, kv, Xn_d
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # ---- derived figures
    pk, src = peaks()
    hbm = float(pk["hbm_gbs"])
    tc_peak = float(pk["bf16_tflops_sustained"] if "bf16_tflops_sustained" in pk else pk["bf16_tflops"])
    step_ms = ms / steps
    blocks = aggregate_blocks_per_s(world, B, steps, ms)
    per_kernel = {s["name"]: {"launches": s["launches"], "ms_per_step": s["ms"] / steps,
                              "gbs": (s["bytes"] / (s["ms"] * 1e-3) / 1e9) if s["bytes"] > 0 else None,
                              "tflops": (s["flops"] / (s["ms"] * 1e-3) / 1e12) if s["flops"] > 0 else None}
                  for s in stats}
    inst_ms = sum(s["ms"] for s in stats) / steps
    # attention: algorithmic KV bytes per launch / event-timed launch duration
    att = [s for s in stats if s["name"] == "attention"]
    att_launch = sum(s["launches"] for s in att)
    att_ms = sum(s["ms"] for s in att) / steps
    att_bytes = attention_bytes_per_step(cfg, ctx)
    att_gbs = att_bytes / (att_ms * 1e-3) / 1e9 if att_ms > 0 else None
    attention = {"kernel": "attn_tc_kernel (block attention, one launch per layer)", "bound": "hbm",
                 "achieved": att_gbs, "peak": hbm, "unit": "GB/s",
                 "frac": (att_gbs / hbm) if att_gbs else None, "peak_source": f"{src} hbm_gbs",
                 "traffic": recorded_traffic(wl.name, "attention"),
                 "algorithmic_bytes_per_launch": att_bytes * steps / att_launch if att_launch else None,
                 "bytes_per_context_token": kv_bytes_per_token(cfg),
                 "launches_per_step": att_launch / steps, "ms_per_step": att_ms,
                 "share_of_step": att_ms / step_ms if step_ms > 0 else None}
    # the tcgen05 GEMM family: tensor-bound at >= TENSOR_BOUND_TOKENS rows, else weight streaming
    gemm = [s for s in stats if s["name"] in GEMM_NAMES]
    g_ms = sum(s["ms"] for s in gemm) / steps
    g_bytes = sum(s["bytes"] for s in gemm) / steps
    g_flops = sum(s["flops"] for s in gemm) / steps
    g_launch = sum(s["launches"] for s in gemm) / steps
    tensor = B * S >= TENSOR_BOUND_TOKENS
    if tensor:
        g_ach, g_peak, g_unit = g_flops / (g_ms * 1e-3) / 1e12, tc_peak, "TFLOP/s"
        g_src = f"{src} bf16_tflops_sustained (kernels inside a long step)"
    else:
        g_ach, g_peak, g_unit = g_bytes / (g_ms * 1e-3) / 1e9, hbm, "GB/s"
        g_src = f"{src} hbm_gbs"
    gemm_roof = {"kernel": "gemm_tc (all tcgen05 GEMM launches of a step)", "bound": "tensor" if tensor else "hbm",
                 "achieved": g_ach, "peak": g_peak, "unit": g_unit, "frac": g_ach / g_peak, "peak_source": g_src,
                 "traffic": recorded_traffic(wl.name, "gemm"),
                 "algorithmic_bytes_per_launch": g_bytes / g_launch, "flops_per_launch": g_flops / g_launch,
                 "launches_per_step": g_launch, "ms_per_step": g_ms,
                 "share_of_step": g_ms / step_ms if step_ms > 0 else None,
                 # per-launch events separate the launches (no PDL overlap): the
                 # summed durations can exceed the step; this bound uses the
                 # step instead
                 "frac_if_step_bounded": (g_ach * g_ms / min(g_ms, step_ms)) / g_peak}
    dominant, second = (attention, gemm_roof) if att_ms >= g_ms else (gemm_roof, attention)
    exp_k = 0.0
    run_p = 1.0
    for q in wl.p_accept[:J]:
        run_p *= q
        exp_k += run_p

    res = {
        "workload": wl.name, "value": blocks, "ms_per_step": step_ms, "steps": steps, "warmup": warmup,
        "desc": workload_desc(wl), "batch": B, "ctx": int(ctx.max()), "ctx_mean": float(ctx.mean()),
        "kv_state": ("drawn (seeded template pages mapped onto the pool)" if wl.kv_fill == "template"
                     else "prefilled through dflash_inject_context"),
        "draft_tokens_per_s": J * blocks, "expected_committed_tokens_per_s": (exp_k + 1) * blocks,
        "mean_accept_len": float(gpu_acc.mean()), "expected_accept_len": exp_k,
        "roofline": dominant, "roofline_second": second, "attention_gbs": att_gbs,
        "per_kernel": per_kernel, "instrumented_ms_per_step": inst_ms,
        "eager_ms_per_step": ms_eager / steps,
        "e2e": {"value": aggregate_blocks_per_s(world, B, steps, ms_e2e), "unit": "blocks/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "per step: H2D of the new tokens' features, anchors and target ids from pinned memory, "
                       "the four C-ABI calls launched eagerly, D2H of accept/bonus/committed, synchronise"
                       + ("; sampling mode: the target logits and uniforms stay resident in HBM (not copied per "
                          "step: in serving they come from the target model on the same GPU)" if sampling else "")},
        "e2e_graph": {"value": aggregate_blocks_per_s(world, B, steps, ms_e2e_graph), "unit": "blocks/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "how": "the same copies around one replay of the captured step"},
        "prefill_injection": prefill_inj, "gpu_launches": launches, "launches_per_step": launches / steps,
        "clocks": clocks, "setup_s": setup_s,
    }

    # ---- CPU baseline: the oracle on a bounded sample (N=1 only)
    if world == 1 and not args.skip_cpu:
        v, el = oracle_request_rate(wl, W, ctx, Xp, cu, Xn, anchor, tgt, templates, table, cpu_reqs)
        res["cpu_baseline"] = {
            "value": v, "unit": "blocks/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"one full drafting step (inject {S} tokens, forward, top-16, select, verify) of each of "
                      f"requests {cpu_reqs} of {B}: {el:.1f} s of fp64 numpy on the host; blocks/s extrapolated "
                      f"linearly to the batch (requests are independent); oracle KV set-up untimed"}
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    from block_diffusion_drafter_context_gb300.build import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
    build()

    head = bench_workload(args.workload, args.layers, args.batch, args.ctx, args.vocab)
    extras = [] if (world > 1 or args.extra in ("", "none")) else [
        n for n in args.extra.split(",") if n and n != args.workload]
    res = run_workload(args, head, args.steps, args.warmup, world, local, dev, headline=True)
    others = {}
    for n in extras:
        try:
            others[n] = run_workload(args, bench_workload(n), args.extra_steps, 3, world, local, dev,
                                     headline=False)
        except Exception as e:   # reported, never fatal to the headline line
            others[n] = {"error": f"{type(e).__name__}: {e}"}
    cpu = res.get("cpu_baseline")
    if cpu is not None and not args.skip_cpu:
        cpu["single_thread"] = single_thread_oracle()

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return

    cfg = head.cfg
    line = {
        "metric": metric(cfg), "value": res["value"], "unit": "blocks/s", "n_gpus": world, "steps": args.steps,
        "mode": "sampling (T=1 path sampling, rejection verification)" if args.mode == "sampling" else "greedy",
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": res["desc"], "batch": res["batch"], "ctx": res["ctx"],
                   "l2": f"no flush: every step streams {weight_bytes(cfg) / 1e9:.1f} GB of drafter weights"
                         + (f" and {attention_bytes_per_step(cfg, [res['ctx_mean']] * res['batch']) / 1e9:.1f} GB"
                            f" of draft KV" if head.batch > 1 else "") + ", > 129 MB L2",
                   "kv_state": res["kv_state"],
                   "weights": "fp8-e4m3 + fp32 row scales (activations bf16)" if cfg.weight_fp8 else cfg.dtype,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": res["roofline"],
        "roofline_second": res["roofline_second"],
        "attention": {"gbs": res["attention_gbs"], "frac": res["roofline"]["frac"]
                      if res["roofline"]["kernel"].startswith("attn") else res["roofline_second"]["frac"]},
        "cpu_baseline": res.get("cpu_baseline"),
        "e2e": res["e2e"], "e2e_graph": res["e2e_graph"],
        "gpu_launches": res["gpu_launches"], "launches_per_step": res["launches_per_step"],
        "clocks": res["clocks"], "gemm_pairs": bool(args.gemm_pairs), "fused_topk": bool(args.fused_topk),
    }
    for k in ("draft_tokens_per_s", "expected_committed_tokens_per_s", "mean_accept_len", "expected_accept_len",
              "per_kernel", "instrumented_ms_per_step", "eager_ms_per_step", "prefill_injection", "setup_s"):
        line[k] = res[k]
    if others:
        line["other_workloads"] = {
            n: (o if "error" in o else {
                "workload": o["desc"], "value": o["value"], "unit": "blocks/s", "ms_per_step": o["ms_per_step"],
                "steps": o["steps"], "kv_state": o["kv_state"], "e2e": o["e2e"]["value"],
                "e2e_graph": o["e2e_graph"]["value"], "roofline": o["roofline"], "roofline_second": o["roofline_second"],
                "attention_gbs": o["attention_gbs"], "eager_ms_per_step": o["eager_ms_per_step"],
                "per_kernel": o["per_kernel"], "prefill_injection": o["prefill_injection"],
                "cpu_baseline": o.get("cpu_baseline"), "gpu_launches": o["gpu_launches"]})
            for n, o in others.items()}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--extra", default=DEFAULT_EXTRA,
                    help="other workloads measured after the headline one (N=1), or 'none'")
    ap.add_argument("--extra-steps", type=int, default=10)
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--mode", default="greedy", choices=["greedy", "sampling"],
                    help="path selection and verification: greedy (default) or sampling + rejection")
    ap.add_argument("--oracle-probe", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--fused-topk", type=int, default=0,
                    help="LM head with its top-16 epilogue (1) or logits + standalone top-16 (0, default)")
    ap.add_argument("--gemm-pairs", type=int, default=1,
                    help="256-token GEMM tiles on CTA pairs with the 2-SM MMA where the plan favours it "
                         "(1, default) or always on single CTAs (0)")
    # smaller variants of the headline workload for profiling captures
    ap.add_argument("--layers", type=int, default=None, help="drafter layers (profiling cases)")
    ap.add_argument("--batch", type=int, default=None, help="requests (profiling cases)")
    ap.add_argument("--ctx", type=lambda s: tuple(int(x) for x in s.split(",")), default=None,
                    help="context lengths lo,hi (profiling cases)")
    ap.add_argument("--vocab", type=int, default=None, help="vocabulary (profiling cases)")
    args = ap.parse_args()
    if args.oracle_probe:
        print(json.dumps(oracle_probe(args.oracle_probe)), flush=True)
        return
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args, bench_workload(args.workload, args.layers, args.batch, args.ctx, args.vocab))
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
