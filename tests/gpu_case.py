"""Shared set-up for the GPU parity tests: one synthetic workload on the
device (weights, paged KV cache filled by the library's own injection) and
the fp64 oracle's view of the same inputs."""
from __future__ import annotations

import functools

import numpy as np

import oracle as O
from synthetic import WORKLOADS, gen

TOL = {"bf16": 2e-2, "f32": 1e-4}


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def to_np(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy() if t.is_floating_point() else t.cpu().numpy()


class Case:
    """A workload prefilled on the GPU through dflash_inject_context."""

    def __init__(self, name: str, device: str = "cuda", gemm_ctas: int = 0, per_request: bool = False):
        import torch
        from block_diffusion_drafter_context_gb300 import binding as Bd
        from block_diffusion_drafter_context_gb300.drafter import Drafter, PagedKV, to_device
        self.torch = torch
        self.to_device = to_device
        wl = WORKLOADS[name]
        self.wl, self.cfg = wl, wl.cfg
        cfg = self.cfg
        self.W = gen.make_weights(cfg, wl.seed)
        self.ctx = gen.context_lengths(wl)
        self.B = len(self.ctx)
        self.table, self.npages = gen.page_table(self.ctx + cfg.block, cfg.page_size, wl.seed)
        self.template = wl.kv_fill == "template"
        self.X = None if self.template else gen.target_hidden(cfg, int(self.ctx.sum()), wl.seed, "prefill")
        self.cu = np.concatenate([[0], np.cumsum(self.ctx)]).astype(np.int32)
        self.anchor = gen.anchors(wl)
        self.device = device
        self.per_request = per_request
        prefill = 0 if self.template else int(self.ctx.max() if per_request else self.ctx.sum())
        self.dr = Drafter(cfg, self.W, max_batch=self.B, max_new_tokens=max(16 * self.B, prefill), device=device)
        if gemm_ctas:
            Bd.dflash_set_gemm_ctas(self.dr.ctx, gemm_ctas)
        self.kv = PagedKV(cfg, self.table, self.npages, device=device)
        self.ctx_d = torch.zeros(self.B, dtype=torch.int32, device=device)
        if self.template:
            # drawn cache state: template pages mapped onto the pool
            self.tk, self.tv = gen.kv_templates(cfg, wl.kv_templates, wl.seed)
            self.pmap = gen.kv_page_map(cfg, self.npages, wl.kv_templates, wl.seed)
            self.kv.fill_from_templates(self.tk, self.tv, self.pmap)
            self.ctx_d.copy_(to_device(self.ctx, device))
        elif per_request:
            # one injection call per request, through a view of its page-table row
            zero = torch.zeros(1, dtype=torch.int32, device=device)
            for b in range(self.B):
                if self.ctx[b] == 0:
                    continue
                cu1 = to_device(np.array([0, self.ctx[b]], np.int32), device)
                Bd.dflash_inject_context(self.dr.ctx, self.kv.row(b), to_device(self.X[self.cu[b]:self.cu[b + 1]], device),
                                         cu1, int(self.ctx[b]), zero, self.ctx_d[b:b + 1], 1, self.dr.workspace,
                                         self.dr.ws_bytes, None)
        elif self.ctx.sum() > 0:
            self.dr.inject_context(self.kv, to_device(self.X, device), to_device(self.cu, device), self.ctx_d)
        self.anchor_d = to_device(self.anchor, device)
        torch.cuda.synchronize()

    # ---- oracle side
    @functools.lru_cache(maxsize=None)
    def oracle_kv(self, b: int):
        n = int(self.ctx[b])
        if n == 0:
            z = np.zeros((0, self.cfg.n_kv_heads, self.cfg.head_dim))
            return [(z, z) for _ in range(self.cfg.n_layers)]
        if self.template:
            return [(O.f64(k), O.f64(v)) for k, v in
                    gen.template_request_kv(self.cfg, self.tk, self.tv, self.pmap, self.table[b], n)]
        return O.inject_context(self.cfg, self.W, self.X[self.cu[b]:self.cu[b + 1]], np.arange(n))

    @functools.lru_cache(maxsize=None)
    def oracle_draft(self, b: int):
        return O.draft_request(self.cfg, self.W, self.oracle_kv(b), int(self.ctx[b]), int(self.anchor[b]))

    # ---- device side
    def gpu_kv(self, b: int, layer: int, n: int | None = None):
        n = int(self.ctx[b]) if n is None else n
        npg = (n + 63) // 64
        pages = self.torch.as_tensor(self.table[b, :npg].astype(np.int64), device=self.device)
        k = self.kv.k[layer][pages].permute(0, 2, 1, 3).reshape(npg * 64, self.cfg.n_kv_heads, -1)[:n]
        # V pages are stored transposed: [page][nkv][d][slot]
        v = self.kv.v[layer][pages].permute(0, 3, 1, 2).reshape(npg * 64, self.cfg.n_kv_heads, -1)[:n]
        return to_np(k), to_np(v)

    def draft(self, want_logits=True):
        return self.dr.draft_block(self.kv, self.ctx_d, self.anchor_d, want_logits=want_logits)
