"""Seeded synthetic inputs for the DFlash drafting workloads.

Everything here is input preparation: random draws, rounding to the storage
type, request lengths, page tables, synthetic target tokens.  None of the
drafting arithmetic (projections, norms, attention, selection, verification)
lives in this module; the oracle and the CUDA path each implement that on
their own and receive these arrays as inputs.

Determinism: every array is drawn from numpy's Philox counter-based
generator keyed by (seed, array name, chunk index), so results do not depend
on the thread count used to produce them and any chunk can be regenerated
alone.

Storage: bf16 matrices are returned as ``uint16`` arrays of bf16 bit
patterns (round-to-nearest-even from the fp32 draw); fp32 configs return
``float32`` arrays.  Norm gains and biases are always ``float32``.  With
``weight_fp8`` the GEMM weight matrices are ``FP8Weight`` objects: OCP FP8
E4M3 codes with one fp32 scale per row, quantised from the fp32 draw.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _gen(seed: int, name: str, chunk: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), zlib.crc32(name.encode()), int(chunk)])
    return np.random.Generator(np.random.Philox(ss))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(shape, std: float, seed: int, name: str, dtype: str = "f32") -> np.ndarray:
    """N(0, std^2) draws of ``shape``; dtype "bf16" returns rounded bf16 bits."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(ci: int) -> None:
        lo = ci * CHUNK
        hi = min(n, lo + CHUNK)
        v = _gen(seed, name, ci).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if dtype == "bf16":
            out[lo:hi] = f32_to_bf16_bits(v)
        else:
            out[lo:hi] = v

    if nchunks <= 1:
        for ci in range(nchunks):
            work(ci)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


class FP8Weight:
    """A weight matrix W[n][k] = scale[n] * e4m3(codes[n][k]) (OCP FP8 E4M3
    codes, one fp32 scale per row).  A container only: decoding belongs to
    whoever consumes the weights."""

    def __init__(self, codes: np.ndarray, scale: np.ndarray):
        self.codes = np.ascontiguousarray(codes, dtype=np.uint8)
        self.scale = np.ascontiguousarray(scale, dtype=np.float32)
        assert self.codes.ndim == 2 and self.scale.shape == (self.codes.shape[0],)

    @property
    def shape(self):
        return self.codes.shape


def _e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code (ties to even) of fp32 values with |x| <= 448.
    Normal range (|x| >= 2^-6): round the fp32 mantissa to 3 bits and re-bias
    the exponent (127 -> 7); below it, multiples of 2^-9 (subnormal codes)."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    sign = ((u >> np.uint32(24)) & np.uint32(0x80)).astype(np.uint8)
    mag = u & np.uint32(0x7FFFFFFF)
    # normal: round to 3 mantissa bits, nearest even
    r = mag + np.uint32(0x7FFFF) + ((mag >> np.uint32(20)) & np.uint32(1))
    e = (r >> np.uint32(23)).astype(np.int32) - 127 + 7
    m = ((r >> np.uint32(20)) & np.uint32(7)).astype(np.int32)
    normal_code = np.minimum((e << 3) | m, 0x7E)
    # subnormal: |x| / 2^-9 rounded to the nearest integer, ties to even (8 = 2^-6, the first normal code)
    sub_code = np.rint(np.abs(x).astype(np.float64) * 512.0).astype(np.int32)
    code = np.where(mag >= np.uint32(0x3C800000), normal_code, sub_code)   # 0x3C800000 = 2^-6
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def quantize_fp8_rows(w: np.ndarray, plant_all_codes: bool = False) -> FP8Weight:
    """Per-row E4M3 quantisation of a weight matrix (stored bf16 bits or fp32):
    scale[n] = max_k |w[n][k]| / 448, codes = nearest E4M3 of w / scale.
    plant_all_codes: row 0 starts with every finite code (0x00..0x7E,
    0x80..0xFE), so that a kernel meets each one (needs K >= 254)."""
    w = np.asarray(w)
    wf = bf16_bits_to_f32(w) if w.dtype == np.uint16 else np.asarray(w, dtype=np.float32)
    amax = np.abs(wf).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = np.empty(wf.shape, dtype=np.uint8)
    step = max(1, (1 << 24) // max(1, wf.shape[1]))

    def work(r0: int) -> None:
        r1 = min(wf.shape[0], r0 + step)
        x = np.clip(wf[r0:r1] / scale[r0:r1, None], -448.0, 448.0).astype(np.float32)
        codes[r0:r1] = _e4m3_encode(x)

    starts = list(range(0, wf.shape[0], step))
    if len(starts) <= 1:
        for r0 in starts:
            work(r0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    if plant_all_codes:
        allc = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
        assert wf.shape[1] >= len(allc)
        codes[0, :len(allc)] = allc
    return FP8Weight(codes, scale)


def gain(n: int, seed: int, name: str) -> np.ndarray:
    """RMSNorm gain 1 + 0.1*N(0,1): a kernel that ignores the gain fails parity."""
    return (1.0 + 0.1 * normal((n,), 1.0, seed, name)).astype(np.float32)


CONV_SITES = ("pre_attn", "post_attn", "pre_ffn", "post_ffn")


def make_weights(cfg, seed: int) -> dict:
    """Random-init drafter weights, N(0, 1/fan_in), stored in ``cfg.dtype``.

    Layout (row-major, ``y = W x`` with W[out, in]):
      w_fc [H, n_sel*H_t], g_fc [H]; embed [V, H]; lm_head [V, H]; g_final [H]
      layers[l]: g_attn [H], w_q [nq*d, H], w_k [nkv*d, H], w_v [nkv*d, H],
                 g_q [d], g_k [d], w_o [H, nq*d], g_ffn [H],
                 w_gate [F, H], w_up [F, H], w_down [H, F],
                 conv[site] = (w [2*H/16, H], b [2*H/16])   (use_conv only)
      sel: e256 [V, 256], a [r, 256], b [r, 256], w_g [H], b_g ()   (use_selector only)
    """
    dt = cfg.dtype
    H, d, F, V = cfg.hidden, cfg.head_dim, cfg.ffn, cfg.vocab
    nq, nkv = cfg.n_q_heads, cfg.n_kv_heads
    W = {
        "w_fc": normal((H, cfg.feat_in), cfg.feat_in ** -0.5, seed, "w_fc", dt),
        "g_fc": gain(H, seed, "g_fc"),
        "embed": normal((V, H), 1.0, seed, "embed", dt),
        "lm_head": normal((V, H), H ** -0.5, seed, "lm_head", dt),
        "g_final": gain(H, seed, "g_final"),
        "layers": [],
    }
    for l in range(cfg.n_layers):
        p = f"L{l}."
        lw = {
            "g_attn": gain(H, seed, p + "g_attn"),
            "w_q": normal((nq * d, H), H ** -0.5, seed, p + "w_q", dt),
            "w_k": normal((nkv * d, H), H ** -0.5, seed, p + "w_k", dt),
            "w_v": normal((nkv * d, H), H ** -0.5, seed, p + "w_v", dt),
            "g_q": gain(d, seed, p + "g_q"),
            "g_k": gain(d, seed, p + "g_k"),
            "w_o": normal((H, nq * d), (nq * d) ** -0.5, seed, p + "w_o", dt),
            "g_ffn": gain(H, seed, p + "g_ffn"),
            "w_gate": normal((F, H), H ** -0.5, seed, p + "w_gate", dt),
            "w_up": normal((F, H), H ** -0.5, seed, p + "w_up", dt),
            "w_down": normal((H, F), F ** -0.5, seed, p + "w_down", dt),
        }
        if cfg.use_conv:
            G2 = 2 * cfg.conv_groups
            lw["conv"] = {
                s: (normal((G2, H), H ** -0.5, seed, p + "conv." + s + ".w", dt),
                    (0.1 * normal((G2,), 1.0, seed, p + "conv." + s + ".b")).astype(np.float32))
                for s in CONV_SITES
            }
        W["layers"].append(lw)
    if cfg.use_selector:
        E, r = cfg.sel_dim, cfg.sel_rank
        std = (E * r ** 0.5) ** -0.5   # keeps u(p).w(c) near unit scale
        W["sel"] = {
            "e256": normal((V, E), 1.0, seed, "sel.e256", dt),
            "a": normal((r, E), std, seed, "sel.a", dt),
            "b": normal((r, E), std, seed, "sel.b", dt),
            "w_g": normal((H,), H ** -0.5, seed, "sel.w_g"),
            "b_g": np.float32(0.1),
        }
    if getattr(cfg, "weight_fp8", False):
        # every GEMM weight as E4M3 codes + row scales; the embedding and the
        # selector tables stay in dtype.  Small shapes plant every code into
        # row 0 of the first layer's W_q and of the LM head.
        plant = cfg.hidden >= 254
        W["w_fc"] = quantize_fp8_rows(W["w_fc"])
        W["lm_head"] = quantize_fp8_rows(W["lm_head"], plant_all_codes=plant and cfg.vocab <= 4096)
        for l, lw in enumerate(W["layers"]):
            for k in ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down"):
                lw[k] = quantize_fp8_rows(lw[k], plant_all_codes=plant and l == 0 and k == "w_q")
            if "conv" in lw:
                lw["conv"] = {s: (quantize_fp8_rows(w), b) for s, (w, b) in lw["conv"].items()}
    return W


def context_lengths(wl) -> np.ndarray:
    if wl.explicit_ctx is not None:
        return np.asarray(wl.explicit_ctx, dtype=np.int32)
    g = _gen(wl.seed, "ctx_len", 0)
    return g.integers(wl.ctx_lo, wl.ctx_hi + 1, size=wl.batch).astype(np.int32)


def anchors(wl, step: int = 0) -> np.ndarray:
    g = _gen(wl.seed, "anchor", step)
    return g.integers(0, wl.cfg.vocab - 1, size=wl.batch).astype(np.int32)


def target_hidden(cfg, n_tokens: int, seed: int, name: str) -> np.ndarray:
    """Concatenated target hidden states [n_tokens, n_sel*H_t], N(0,1)."""
    return normal((n_tokens, cfg.feat_in), 1.0, seed, "X." + name, cfg.dtype)


def page_table(ctx_capacity: np.ndarray, page_size: int, seed: int):
    """Random page assignment: returns (table [B, max_pages] int32, num_pages).

    Request b owns ceil(cap_b / page_size) pages drawn from a seeded random
    permutation of the pool, so page indirection is exercised.  Unused table
    entries are -1 and are never read by a correct kernel.
    """
    cap = np.asarray(ctx_capacity, dtype=np.int64)
    npg = (cap + page_size - 1) // page_size
    total = int(npg.sum())
    maxp = max(1, int(npg.max()) if len(npg) else 1)
    perm = _gen(seed, "pages", 0).permutation(total).astype(np.int32)
    tab = np.full((len(cap), maxp), -1, dtype=np.int32)
    o = 0
    for b, k in enumerate(npg):
        tab[b, :k] = perm[o:o + k]
        o += k
    return tab, total


def kv_templates(cfg, n_templates: int, seed: int):
    """Template KV pages for a drawn cache state: (K, V), each
    [L][n_templates][nkv][page][d], N(0,1) entries in cfg.dtype."""
    shape = (cfg.n_layers, n_templates, cfg.n_kv_heads, cfg.page_size, cfg.head_dim)
    return (normal(shape, 1.0, seed, "kv_tmpl.k", cfg.dtype), normal(shape, 1.0, seed, "kv_tmpl.v", cfg.dtype))


def kv_page_map(cfg, num_pages: int, n_templates: int, seed: int) -> np.ndarray:
    """[L][num_pages] int32: the template page each pool page of each layer holds."""
    g = _gen(seed, "kv_page_map", 0)
    return g.integers(0, n_templates, size=(cfg.n_layers, num_pages)).astype(np.int32)


def template_request_kv(cfg, tk, tv, page_map, table_row, n: int):
    """Stored (K, V) [n, nkv, d] per layer of a request whose context is a
    drawn cache state: token t sits in slot t % page of pool page
    table_row[t // page], which holds template page page_map[l, page]."""
    t = np.arange(n)
    page = np.asarray(table_row)[t // cfg.page_size]
    out = []
    for l in range(cfg.n_layers):
        tm = page_map[l][page]
        out.append((tk[l][tm, :, t % cfg.page_size, :], tv[l][tm, :, t % cfg.page_size, :]))
    return out


def target_ids(draft: np.ndarray, p_accept, vocab: int, seed: int, step: int = 0) -> np.ndarray:
    """Synthetic target tokens [B, 16] for greedy verification.

    Position i (0-based, < 15) equals draft[:, i] with probability p_accept[i],
    otherwise it is uniform over the vocabulary minus draft[:, i].  The last
    position (the bonus after a fully accepted block) is uniform.
    """
    draft = np.asarray(draft, dtype=np.int64)
    B, S1 = draft.shape
    g = _gen(seed, "target_ids", step)
    u = g.random((B, S1))
    alt = g.integers(0, vocab - 1, size=(B, S1))
    alt = alt + (alt >= draft)
    t = np.where(u < np.asarray(p_accept)[None, :S1], draft, alt)
    last = g.integers(0, vocab, size=(B, 1))
    return np.concatenate([t, last], axis=1).astype(np.int32)
