"""Host-side convenience around the C ABI: weight upload/packing into the
layouts include/dflash.h expects, the paged KV cache, the workspace, and a
``Drafter`` object whose methods call the four entry points.

Marshalling only: packing is concatenation / interleaving of weight rows; all
drafting arithmetic happens in libdflash.
"""
from __future__ import annotations

import numpy as np

from . import binding as B


def _torch():
    import torch
    return torch


def _is_fp8(a) -> bool:
    return hasattr(a, "codes") and hasattr(a, "scale")


def to_device(a, device="cuda"):
    """numpy -> device tensor; uint16 arrays are bf16 bit patterns."""
    torch = _torch()
    if isinstance(a, torch.Tensor):
        return a.to(device)
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    if a.dtype in (np.int32, np.int64):
        return torch.from_numpy(a.astype(np.int32)).to(device)
    return torch.from_numpy(a.astype(np.float32)).to(device)


def make_config(cfg) -> B.dflash_config:
    c = B.dflash_config()
    c.dtype = B.DFLASH_F32 if cfg.dtype == "f32" else B.DFLASH_BF16
    for k in ("hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
              "target_hidden", "n_target_layers", "sel_rank", "sel_dim", "page_size"):
        setattr(c, k, int(getattr(cfg, k)))
    c.block_size = int(cfg.block)
    c.top_k = int(cfg.top_k)
    c.use_conv = int(bool(cfg.use_conv))
    c.use_selector = int(bool(cfg.use_selector))
    c.qk_norm = int(bool(cfg.qk_norm))
    c.fc_norm = int(bool(cfg.fc_norm))
    c.split_act = int(bool(getattr(cfg, "split_act", True)))
    c.mask_id = int(cfg.mask_id)
    c.rope_base = float(cfg.rope_base)
    c.eps = float(cfg.eps)
    c.weight_fp8 = int(bool(getattr(cfg, "weight_fp8", False)))
    return c


CONV_SITES = ("pre_attn", "post_attn", "pre_ffn", "post_ffn")


def fp8_bf16_copies(dw: dict) -> None:
    """bf16 copies of every packed FP8 matrix (the codes' exact values, made by
    the library on the device; the row scales stay in s_*), stored beside them
    under *_bf16: the drafter uses them for its tensor-bound launches (128+
    tokens per launch)."""
    torch = _torch()

    def conv(codes, scale):
        out = torch.empty(codes.shape, dtype=torch.bfloat16, device=codes.device)
        B.dflash_fp8_weights_to_bf16(codes, codes.shape[0], codes.shape[1], out)
        return out

    dw["w_fc_bf16"] = conv(dw["w_fc"], dw["s_fc"])
    dw["lm_head_bf16"] = conv(dw["lm_head"], dw["s_lm_head"])
    for L in dw["layers"]:
        for k, sk in (("w_qkv", "s_qkv"), ("w_o", "s_o"), ("w_gu", "s_gu"), ("w_down", "s_down")):
            L[k + "_bf16"] = conv(L[k], L[sk])
        if "s_conv" in L:
            L["w_conv_bf16"] = [conv(w, sc) for w, sc in zip(L["w_conv"], L["s_conv"])]
    torch.cuda.synchronize()


def upload_weights(cfg, W: dict, device="cuda") -> dict:
    """Upload a weight dict (layout of the synthetic generator) and pack it:
    w_qkv = [w_q; w_k; w_v] rows; w_gu rows interleaved gate_i, up_i; each
    short-conv site's [a; b] coefficient rows (and biases) interleaved per
    channel group, a_g, b_g.  FP8 weights upload their codes (uint8) and put
    the row scales under s_*."""
    torch = _torch()

    def d(a):
        if _is_fp8(a):
            return torch.from_numpy(a.codes).to(device)
        return to_device(a, device)

    def sc(a):
        return torch.from_numpy(a.scale).to(device) if _is_fp8(a) else None

    def rows_cat(parts):
        return torch.cat(parts, 0).contiguous()

    def interleave(a, b):
        return torch.stack([a, b], 1).reshape(2 * a.shape[0], *a.shape[1:]).contiguous()

    def interleave_halves(t):
        """[a; b] rows (first half a, second half b) -> a_0, b_0, a_1, b_1, ..."""
        h = t.shape[0] // 2
        return interleave(t[:h], t[h:])

    out = {k: d(W[k]) for k in ("w_fc", "g_fc", "embed", "lm_head", "g_final")}
    fp8 = _is_fp8(W["lm_head"])
    if fp8:
        out["s_fc"], out["s_lm_head"] = sc(W["w_fc"]), sc(W["lm_head"])
    out["layers"] = []
    for lw in W["layers"]:
        gate, up = d(lw["w_gate"]), d(lw["w_up"])
        L = {
            "g_attn": d(lw["g_attn"]),
            "w_qkv": rows_cat([d(lw["w_q"]), d(lw["w_k"]), d(lw["w_v"])]),
            "g_q": d(lw["g_q"]), "g_k": d(lw["g_k"]), "w_o": d(lw["w_o"]), "g_ffn": d(lw["g_ffn"]),
            "w_gu": interleave(gate, up),
            "w_down": d(lw["w_down"]),
        }
        del gate, up
        if fp8:
            L["s_qkv"] = rows_cat([sc(lw["w_q"]), sc(lw["w_k"]), sc(lw["w_v"])])
            L["s_o"], L["s_down"] = sc(lw["w_o"]), sc(lw["w_down"])
            L["s_gu"] = interleave(sc(lw["w_gate"]), sc(lw["w_up"]))
        if "conv" in lw:
            L["w_conv"] = [interleave_halves(d(lw["conv"][s][0])) for s in CONV_SITES]
            L["b_conv"] = [interleave_halves(d(lw["conv"][s][1])) for s in CONV_SITES]
            if fp8:
                L["s_conv"] = [interleave_halves(sc(lw["conv"][s][0])) for s in CONV_SITES]
        out["layers"].append(L)
    if "sel" in W:
        s = W["sel"]
        out["sel"] = {"e256": d(s["e256"]), "a": d(s["a"]), "b": d(s["b"]), "w_g": d(s["w_g"]),
                      "b_g": float(s["b_g"])}
    return out


def make_weights_struct(dw: dict):
    lay = (B.dflash_layer_weights * len(dw["layers"]))()
    for i, L in enumerate(dw["layers"]):
        s = lay[i]
        for k in ("g_attn", "w_qkv", "g_q", "g_k", "w_o", "g_ffn", "w_gu", "w_down"):
            setattr(s, k, L[k].data_ptr())
        if "w_conv" in L:
            for j in range(4):
                s.w_conv[j] = L["w_conv"][j].data_ptr()
                s.b_conv[j] = L["b_conv"][j].data_ptr()
                if "s_conv" in L:
                    s.s_conv[j] = L["s_conv"][j].data_ptr()
        for k in ("s_qkv", "s_o", "s_gu", "s_down", "w_qkv_bf16", "w_o_bf16", "w_gu_bf16", "w_down_bf16"):
            if k in L:
                setattr(s, k, L[k].data_ptr())
        if "w_conv_bf16" in L:
            for j in range(4):
                s.w_conv_bf16[j] = L["w_conv_bf16"][j].data_ptr()
    w = B.dflash_weights()
    for k in ("w_fc", "g_fc", "embed", "lm_head", "g_final"):
        setattr(w, k, dw[k].data_ptr())
    for k in ("s_fc", "s_lm_head", "w_fc_bf16", "lm_head_bf16"):
        if k in dw:
            setattr(w, k, dw[k].data_ptr())
    w.layers = lay
    if "sel" in dw:
        w.sel_e256 = dw["sel"]["e256"].data_ptr()
        w.sel_a = dw["sel"]["a"].data_ptr()
        w.sel_b = dw["sel"]["b"].data_ptr()
        w.sel_w_g = dw["sel"]["w_g"].data_ptr()
        w.sel_b_g = dw["sel"]["b_g"]
    return w, lay


class PagedKV:
    """Device KV pools (K [L][num_pages][nkv][64][d], V [L][num_pages][nkv][d][64])
    and the page table; zero-filled (slots past a request's length stay finite)."""

    def __init__(self, cfg, page_table: np.ndarray, num_pages: int, device="cuda", zero=True):
        torch = _torch()
        dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
        shape = (cfg.n_layers, num_pages, cfg.n_kv_heads, cfg.page_size, cfg.head_dim)
        vshape = (cfg.n_layers, num_pages, cfg.n_kv_heads, cfg.head_dim, cfg.page_size)
        alloc = torch.zeros if zero else torch.empty
        self.k = alloc(shape, dtype=dt, device=device)
        self.v = alloc(vshape, dtype=dt, device=device)
        self.page_table = to_device(np.ascontiguousarray(page_table, dtype=np.int32), device)
        self.num_pages = int(num_pages)
        self.max_pages = int(page_table.shape[1])
        self.struct = B.dflash_kv(self.k.data_ptr(), self.v.data_ptr(), self.page_table.data_ptr(),
                                  self.num_pages, self.max_pages)

    def fill_from_templates(self, tk: np.ndarray, tv: np.ndarray, page_map: np.ndarray):
        """Set a drawn cache state: pool page p of layer l takes template page
        page_map[l, p] of tk / tv ([L][T][nkv][page][d]); V is stored
        transposed like every V page.  Set-up only (device copies)."""
        torch = _torch()
        dev = self.k.device
        for l in range(self.k.shape[0]):
            idx = torch.from_numpy(page_map[l].astype(np.int64)).to(dev)
            kt = to_device(tk[l], dev).to(self.k.dtype)
            vt = to_device(tv[l], dev).to(self.v.dtype).transpose(2, 3).contiguous()
            self.k[l].copy_(kt.index_select(0, idx))
            self.v[l].copy_(vt.index_select(0, idx))
            del kt, vt

    def row(self, b: int) -> B.dflash_kv:
        """dflash_kv whose page table is request b's row alone (a batch of one)."""
        r = self.page_table[b:b + 1]
        return B.dflash_kv(self.k.data_ptr(), self.v.data_ptr(), r.data_ptr(), self.num_pages, self.max_pages)


class Drafter:
    """One drafter context: uploaded weights, a workspace, the C handle."""

    def __init__(self, cfg, W: dict, max_batch: int, max_new_tokens: int, device="cuda", dev_weights=None,
                 fp8_copies: bool = True):
        """fp8_copies (FP8 weights only): also keep bf16 copies of the matrices
        for the launches of 128+ tokens, where bf16 weights are faster."""
        torch = _torch()
        self.cfg = cfg
        self.dw = dev_weights if dev_weights is not None else upload_weights(cfg, W, device)
        if getattr(cfg, "weight_fp8", False) and fp8_copies and "w_fc_bf16" not in self.dw:
            fp8_bf16_copies(self.dw)
        self.wstruct, self._lay = make_weights_struct(self.dw)
        self.cstruct = make_config(cfg)
        self.ctx = B.dflash_create(self.cstruct, self.wstruct)
        self.ws_bytes = B.dflash_workspace_bytes(self.ctx, max_batch, max_new_tokens)
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.max_batch, self.max_new_tokens = max_batch, max_new_tokens
        self.device = device
        self.block = int(cfg.block)     # runtime block size S

    def set_block_size(self, block_size: int):
        """Run the next steps at block size S (2..the configured block size)."""
        B.dflash_set_block_size(self.ctx, int(block_size))
        self.block = int(block_size)

    def close(self):
        if getattr(self, "ctx", None):
            B.dflash_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def act_dtype(self):
        torch = _torch()
        return torch.float32 if self.cfg.dtype == "f32" else torch.bfloat16

    def status(self, stream=None) -> int:
        return B.dflash_read_status(self.workspace, stream)

    # ---- the four calls, allocating their outputs with torch
    def inject_context(self, kv: PagedKV, target_hidden, cu_new, ctx_len_in, ctx_len_out=None, stream=None):
        batch = int(cu_new.shape[0]) - 1
        total = int(target_hidden.shape[0])
        if ctx_len_out is None:
            ctx_len_out = ctx_len_in
        B.dflash_inject_context(self.ctx, kv.struct, target_hidden, cu_new, total, ctx_len_in, ctx_len_out,
                                batch, self.workspace, self.ws_bytes, stream)
        return ctx_len_out

    def draft_block(self, kv: PagedKV, ctx_len, anchor_ids, want_logits=False, stream=None):
        torch = _torch()
        b = int(anchor_ids.shape[0])
        dev = self.device
        S = self.block
        out = {
            "topk_ids": torch.empty((b, S - 1, 16), dtype=torch.int32, device=dev),
            "topk_logits": torch.empty((b, S - 1, 16), dtype=torch.float32, device=dev),
            "final_hidden": torch.empty((b, S, self.cfg.hidden), dtype=self.act_dtype, device=dev),
            "logits": torch.empty((b, S - 1, self.cfg.vocab), dtype=torch.float32, device=dev) if want_logits else None,
        }
        B.dflash_draft_block(self.ctx, kv.struct, ctx_len, anchor_ids, b, out["topk_ids"], out["topk_logits"],
                             out["final_hidden"], out["logits"], self.workspace, self.ws_bytes, stream)
        return out

    def select_path(self, anchor_ids, topk_ids, topk_logits, final_hidden, want_scores=True, stream=None):
        torch = _torch()
        b = int(topk_ids.shape[0])
        J = self.block - 1
        draft = torch.empty((b, J), dtype=torch.int32, device=self.device)
        scores = (torch.empty((b, J, 16, 16), dtype=torch.float32, device=self.device)
                  if (want_scores and self.cfg.use_selector) else None)
        B.dflash_select_path(self.ctx, anchor_ids, topk_ids, topk_logits, final_hidden, b, draft, scores,
                             self.workspace, self.ws_bytes, stream)
        return draft, scores

    def sample_path(self, anchor_ids, topk_ids, topk_logits, final_hidden, temperature, uniforms, stream=None):
        """Draft drawn over the path scores at a temperature: (draft [b,J], q [b,J,16])."""
        torch = _torch()
        b = int(topk_ids.shape[0])
        J = self.block - 1
        draft = torch.empty((b, J), dtype=torch.int32, device=self.device)
        probs = torch.empty((b, J, 16), dtype=torch.float32, device=self.device)
        B.dflash_sample_path(self.ctx, anchor_ids, topk_ids, topk_logits, final_hidden, b, temperature, uniforms,
                             draft, probs, None, self.workspace, self.ws_bytes, stream)
        return draft, probs

    def verify_rejection(self, target_logits, draft_ids, topk_ids, draft_probs, u_accept, u_bonus, stream=None):
        """Rejection-sampling verification: (accept_len, bonus, committed)."""
        torch = _torch()
        b = int(draft_ids.shape[0])
        dev = draft_ids.device
        acc = torch.empty(b, dtype=torch.int32, device=dev)
        bonus = torch.empty(b, dtype=torch.int32, device=dev)
        com = torch.empty((b, self.block), dtype=torch.int32, device=dev)
        B.dflash_verify_rejection(self.ctx, target_logits, draft_ids, topk_ids, draft_probs, u_accept, u_bonus, b,
                                  acc, bonus, com, self.workspace, self.ws_bytes, stream)
        return acc, bonus, com

    @staticmethod
    def verify_greedy(draft_ids, target_ids, stream=None):
        """Greedy prefix acceptance; the block size is target_ids' second extent."""
        torch = _torch()
        b, S = int(target_ids.shape[0]), int(target_ids.shape[1])
        dev = draft_ids.device
        acc = torch.empty(b, dtype=torch.int32, device=dev)
        bonus = torch.empty(b, dtype=torch.int32, device=dev)
        com = torch.empty((b, S), dtype=torch.int32, device=dev)
        B.dflash_verify_greedy(draft_ids, target_ids, b, S, acc, bonus, com, stream)
        return acc, bonus, com
