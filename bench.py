"""Benchmark of one DFlash drafting step on GB300.

A step is the whole hot path for every request of the workload: inject the
S new tokens' target features into every drafter layer's paged KV cache,
draft one S-token block (one forward of the drafter), select the path, and
verify greedily against synthetic target tokens (S = 16 unless the workload
sets a smaller runtime block size).  Default workload: the Qwen3-8B-shaped
drafter (5 layers, hidden 4096, vocab 151936), batch 1, 2048 tokens of
context (configs C2-C4 are parity cases, not bench lines).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload C1|C2|C3|C4|C1S5|C2S5] [--mode greedy|sampling]

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on the same workload instead (the deliberately slow reference arm).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import WORKLOADS, gen  # noqa: E402

METRIC = "drafted blocks/sec (16-tok) at batch×ctx on 1 GB300; attention HBM GB/s"


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


def prefill_injection_flops(cfg, tokens: int) -> float:
    """Dense flops of injecting `tokens` context tokens: the context-feature
    projection [tokens, n_sel*H_t] x [n_sel*H_t, H] and every layer's K and V
    projections [tokens, H] x [H, 2*nkv*d]."""
    return 2.0 * tokens * cfg.hidden * (cfg.feat_in + cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim)


def workload_desc(wl):
    c = wl.cfg
    return (f"{wl.name}: {c.name} drafter (L={c.n_layers}, H={c.hidden}, {c.n_q_heads}q/{c.n_kv_heads}kv x "
            f"{c.head_dim}, F={c.ffn}, V={c.vocab}), batch {wl.batch}, context "
            f"{wl.ctx_lo if wl.ctx_lo == wl.ctx_hi else f'U[{wl.ctx_lo},{wl.ctx_hi}]'}, "
            f"{c.n_target_layers}x{c.target_hidden} target features, block size {c.block}, "
            f"{c.block} new tokens injected per step" + (", FP8 E4M3 weights (per-row scales)" if c.weight_fp8 else ""))


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
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------- inputs
def make_inputs(wl):
    cfg = wl.cfg
    W = gen.make_weights(cfg, wl.seed)
    ctx = gen.context_lengths(wl)
    B = len(ctx)
    table, npages = gen.page_table(ctx + cfg.block, cfg.page_size, wl.seed)
    cu = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    # drawn cache state (template pages) or a prefill through the injection
    Xp = None if wl.kv_fill == "template" else gen.target_hidden(cfg, int(ctx.sum()), wl.seed, "prefill")
    Xn = gen.target_hidden(cfg, cfg.block * B, wl.seed, "step")
    anchor = gen.anchors(wl)
    return W, ctx, table, npages, cu, Xp, Xn, anchor


def kv_templates(wl, npages):
    """(K templates, V templates, page map) of a drawn cache state, else None."""
    if wl.kv_fill != "template":
        return None
    tk, tv = gen.kv_templates(wl.cfg, wl.kv_templates, wl.seed)
    return tk, tv, gen.kv_page_map(wl.cfg, npages, wl.kv_templates, wl.seed)


def run_reference(args, wl):
    """The reference arm: the fp64 oracle on the host cores."""
    W, ctx, table, npages, cu, Xp, Xn, anchor = make_inputs(wl)
    t0 = time.time()
    kvs = oracle_setup(wl, W, ctx, Xp, cu, templates=kv_templates(wl, npages), table=table)
    setup_s = time.time() - t0
    import oracle as O
    first = oracle_step(wl, W, kvs, ctx, Xn, anchor, np.zeros((wl.batch, wl.cfg.block), np.int32),
                        range(wl.batch))
    draft = np.stack([o["draft"] for o in first])
    target = gen.target_ids(draft, wl.p_accept, wl.cfg.vocab, seed=wl.seed)
    for _ in range(args.warmup):
        oracle_step(wl, W, kvs, ctx, Xn, anchor, target, range(wl.batch))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, W, kvs, ctx, Xn, anchor, target, range(wl.batch))
    el = time.perf_counter() - t0
    v = wl.batch * args.steps / el
    cores = blas_threads()
    line = {"impl": "reference", "metric": metric(wl.cfg), "value": v, "unit": "blocks/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(wl), "batch": wl.batch,
                                            "ctx": int(ctx.max())},
            "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} full steps of all {wl.batch} request(s) after "
                                       f"{args.warmup} warm-up; oracle KV prefill ({setup_s:.1f} s) untimed"},
            "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    from block_diffusion_drafter_context_gb300 import binding as Bd
    from block_diffusion_drafter_context_gb300.build import build
    from block_diffusion_drafter_context_gb300.drafter import Drafter, PagedKV, to_device

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
    cfg = wl.cfg
    t_setup = time.time()
    W, ctx, table, npages, cu, Xp, Xn, anchor = make_inputs(wl)
    B, S, J = wl.batch, cfg.block, cfg.block - 1
    prefill = 0 if wl.kv_fill == "template" else int(ctx.max())
    dr = Drafter(cfg, W, max_batch=B, max_new_tokens=max(S * B, prefill), device=dev)
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
    tgt = gen.target_ids(draft.cpu().numpy(), wl.p_accept, cfg.vocab, seed=wl.seed)
    target_d.copy_(torch.from_numpy(tgt))
    setup_s = time.time() - t_setup

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert dr.status() == 0, "device status after warm-up"

    # the step's launches, captured once into a CUDA graph (no host work per launch)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
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

    with ClockSampler(local) as cs:
        cs.mark(True)
        ms = timed(graph.replay, args.steps)
        cs.mark(False)
    clocks = cs.summary()
    ms_eager = timed(step, args.steps)
    assert dr.status() == 0, "device status after the timed region"

    # ---- instrumented pass: CUDA events around every launch, captured with
    # the K steps into one graph so host gaps do not enter the durations
    Bd.dflash_profile_begin(dr.ctx)      # eager pass first: creates the event pool outside capture
    for _ in range(args.steps):
        step()
    stats_eager = Bd.dflash_profile_end(dr.ctx)
    Bd.dflash_profile_begin(dr.ctx)
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prof):
        for _ in range(args.steps):
            step()
    g_prof.replay()
    torch.cuda.synchronize()
    stats = Bd.dflash_profile_end(dr.ctx)
    launches = sum(s["launches"] for s in stats)
    del g_prof

    # ---- end to end through the public API with host buffers
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
    stream = torch.cuda.current_stream()

    def step_e2e():
        x_dev.copy_(pin_x, non_blocking=True)
        anc_d.copy_(pin_a, non_blocking=True)
        if sampling:
            uni_all.copy_(pin_t, non_blocking=True)
            uni_d.view(-1).copy_(uni_all[:B * J], non_blocking=True)
            ua_d.view(-1).copy_(uni_all[B * J:B * 2 * J], non_blocking=True)
            ub_d.copy_(uni_all[B * 2 * J:], non_blocking=True)
        else:
            target_d.copy_(pin_t, non_blocking=True)
        graph.replay()
        out_acc.copy_(acc, non_blocking=True)
        out_bonus.copy_(bonus, non_blocking=True)
        out_com.copy_(com, non_blocking=True)
        stream.synchronize()   # the host reads the step's result before the next step

    for _ in range(2):
        step_e2e()
    ms_e2e = timed(step_e2e, args.steps)
    h2d = pin_x.numel() * pin_x.element_size() + pin_a.numel() * 4 + pin_t.numel() * 4
    d2h = (out_acc.numel() + out_bonus.numel() + out_com.numel()) * 4
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

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return

    pk, src = peaks()
    hbm = float(pk["hbm_gbs"])
    gemm = [s for s in stats if s["name"] in ("fc", "kv_inject", "qkv", "o_proj", "gate_up", "down", "lm_head",
                                             "conv_coef")]
    g_ms = sum(s["ms"] for s in gemm)
    g_bytes = sum(s["bytes"] for s in gemm)
    g_launch = sum(s["launches"] for s in gemm)
    per_kernel = {s["name"]: {"launches": s["launches"], "ms_per_step": s["ms"] / args.steps,
                              "gbs": (s["bytes"] / (s["ms"] * 1e-3) / 1e9) if s["bytes"] > 0 else None}
                  for s in stats}
    att = [s for s in stats if s["name"] == "attention"]
    # K and V read per step: each request's context plus the S tokens this step injected, plus the S block keys
    kv_bytes_step = float(sum(int(c) + 2 * S for c in ctx)) * cfg.n_layers * cfg.n_kv_heads * cfg.head_dim * 2 * 2
    att_ms = sum(s["ms"] for s in att) / args.steps
    att_gbs = kv_bytes_step / (att_ms * 1e-3) / 1e9 if att_ms > 0 else None
    total_ms_inst = sum(s["ms"] for s in stats) / args.steps
    step_ms = ms / args.steps
    blocks = aggregate_blocks_per_s(world, B, args.steps, ms)
    exp_k = 0.0
    run_p = 1.0
    for q in wl.p_accept[:J]:
        run_p *= q
        exp_k += run_p
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        try:
            traffic = json.load(open(tfile)).get(wl.name, {}).get("gemm_bytes_per_launch")
        except Exception:
            traffic = None

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if world == 1 and not args.skip_cpu:
        kvs = oracle_setup(wl, W, ctx, Xp, cu, requests=[0], templates=templates, table=table)
        t0 = time.perf_counter()
        oracle_step(wl, W, kvs, ctx, Xn, anchor, tgt, [0])
        el = time.perf_counter() - t0
        cpu = {"value": 1.0 / el, "unit": "blocks/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"one full drafting step (inject {S} tokens, forward, top-16, select, verify) of request "
                         f"0 of {B}; {el:.1f} s of fp64 numpy on the host; oracle KV prefill untimed"}

    line = {
        "metric": metric(cfg), "value": blocks, "unit": "blocks/s", "n_gpus": world, "steps": args.steps,
        "mode": "sampling (T=1 path sampling, rejection verification)" if sampling else "greedy",
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": workload_desc(wl), "batch": B, "ctx": int(ctx.max()),
                   "l2": f"no flush: every step streams {weight_bytes(cfg) / 1e9:.1f} GB of drafter weights, "
                         f"> 129 MB L2",
                   "weights": "fp8-e4m3 + fp32 row scales (activations bf16)" if cfg.weight_fp8 else cfg.dtype,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "draft_tokens_per_s": J * blocks,
        "expected_committed_tokens_per_s": (exp_k + 1) * blocks,
        "roofline": {"kernel": "gemm_tc (all tcgen05 GEMM launches of a step)", "bound": "hbm",
                     "achieved": g_bytes / (g_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": g_bytes / (g_ms * 1e-3) / 1e9 / hbm, "peak_source": f"{src} hbm_gbs",
                     "traffic": traffic, "algorithmic_bytes_per_launch": g_bytes / g_launch,
                     "launches_per_step": g_launch / args.steps, "share_of_step": g_ms / (total_ms_inst * args.steps)},
        "attention": {"kv_bytes_per_step": kv_bytes_step, "ms_per_step": att_ms, "gbs": att_gbs,
                      "frac": (att_gbs / hbm) if att_gbs else None},
        "per_kernel": per_kernel,
        "instrumented_ms_per_step": total_ms_inst,
        "eager_ms_per_step": ms_eager / args.steps,
        "cpu_baseline": cpu,
        "e2e": {"value": aggregate_blocks_per_s(world, B, args.steps, ms_e2e), "unit": "blocks/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "prefill_injection": prefill_inj,
        "gpu_launches": launches,
        "launches_per_step": launches / args.steps,
        "clocks": clocks,
        "setup_s": setup_s,
    }
    print(json.dumps(line), flush=True)
    dr.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="C1")
    ap.add_argument("--skip-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--mode", default="greedy", choices=["greedy", "sampling"],
                    help="path selection and verification: greedy (default) or sampling + rejection")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
