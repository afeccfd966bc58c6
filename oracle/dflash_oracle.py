"""fp64 CPU oracle for one DFlash block-diffusion drafting step.

TEST INFRASTRUCTURE ONLY.  This module is the independent checker of the CUDA
library: only the test suite, the smoke check and the benchmark's CPU-baseline
leg may import it.  It shares no code with the CUDA path; the only thing the
two sides share is the seeded input data.

It is a plain, slow, direct transcription of what the pages define, in
float64 from the stored (bf16 or fp32) inputs, with no intermediate rounding,
no blocking and no fusion.  numpy matmul, sort and elementwise routines serve
as the library primitives.

Pages the method is taken from (cited below by these tags):
  [DF]   "DFlash - Difusion de Bloques para Decodificacion Especulativa en
         Flash" (gist.science, paper 2602.06036)
  [DF2]  "DFlash 2: optimizacion de la decodificacion especulativa para
         inferencia paralela de LLMs" (kerneldigest.dev)
  [FD]   "FlexDraft" (gist.science, paper 2605.20022)
  [BW]   "DFlash: Avance en la inferencia de LLM con decodificacion
         especulativa en NVIDIA Blackwell" (emedoteme.es)

Readings taken where the pages are silent (each one is listed in the design
notes with its reason):
  * context feature = RMSNorm(W_fc x) with no bias; layer sets are
    concatenated in ascending layer order;
  * the feature enters each layer's own W_k / W_v with no input norm; K gets
    the per-head k-norm and RoPE at its absolute position;
  * drafter layers are pre-norm Qwen3-style: RMSNorm eps 1e-6, per-head q/k
    RMSNorm, SwiGLU FFN, no biases, softmax scale 1/sqrt(d);
  * RoPE pairs (i, i + d/2) with theta_i = base^(-2i/d);
  * the mask token is the last vocabulary row (id V-1);
  * short conv: [a; b] = tanh(W_c y_j + b_c), channel c uses group c // 16,
    out_j = y_j + a_j*y_j + b_j*y_{j-1}, y_{-1} = 0, applied to the normed
    input (pre) and to the sublayer output (post) of attention and FFN;
  * selector: gate g_j = sigmoid(w_g . h_j + b_g) on the final-normed hidden
    state, u(t) = A e256[t], w(t) = B e256[t],
    s_j(p, c) = z_j[c] + g_j * u(p) . w(c), p = anchor for the first mask
    position; greedy path with ties to the lower token id;
  * ties in every top-k / argmax go to the lower token id.

Parity unpinned: the DFlash-2 parameter counts printed by [DF2] (16.5 M
conv, 2.0 M selector) are not reproduced by any reading of the shapes; no
function here depends on them.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# storage decode
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """OCP FP8 E4M3 codes -> float64, from the format's definition (OFP8
    specification, E4M3: sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities).  Normal (E >= 1): (-1)^S * 2^(E-7) * (1 + M/8);
    subnormal (E = 0): (-1)^S * 2^-6 * M/8; S.1111.111 is NaN."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


def f64(a) -> np.ndarray:
    """Stored input -> float64.  uint16 arrays hold bf16 bit patterns; an FP8
    weight (E4M3 codes with one scale per row, "draft quantization") is
    scale[n] * e4m3(codes[n][k])."""
    if hasattr(a, "codes") and hasattr(a, "scale"):
        return e4m3_decode(a.codes) * np.asarray(a.scale, dtype=np.float64)[:, None]
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# --------------------------------------------------------------------------
# building blocks
# --------------------------------------------------------------------------
def rms_norm(x, gain, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: gain * x / sqrt(mean(x^2) + eps).

    Layer internals are not given by the pages; pre-norm RMSNorm is the
    Qwen3-style reading for the Qwen3-shaped drafter.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * f64(gain)


def rope(x, positions, base: float) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing (i, i + d/2).

    x: [T, n_heads, d]; positions: [T] absolute positions.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    theta = float(base) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def softmax(s, axis=-1):
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


# --------------------------------------------------------------------------
# [DF] §2.2 "Diseno de Inferencia": context feature and KV injection
# --------------------------------------------------------------------------
def context_feature(cfg, W, target_hidden) -> np.ndarray:
    """[DF] §2.2, context-feature bullet: the hidden states of a fixed set of
    target layers, concatenated, are projected to a compact target context
    feature.  target_hidden: [T, n_sel*H_t] -> f: [T, H]."""
    f = f64(target_hidden) @ f64(W["w_fc"]).T
    if cfg.fc_norm:
        f = rms_norm(f, W["g_fc"], cfg.eps)
    return f


def inject_layer(cfg, lw, feature, positions):
    """[DF] §2.2, KV-injection bullet (and §3 item 2): the context feature is
    projected by every drafter layer's own K and V projections and kept in
    that layer's KV cache.  Returns K (post k-norm and RoPE) and V, each
    [T, n_kv, d]."""
    T = feature.shape[0]
    nkv, d = cfg.n_kv_heads, cfg.head_dim
    k = (feature @ f64(lw["w_k"]).T).reshape(T, nkv, d)
    if cfg.qk_norm:
        k = rms_norm(k, lw["g_k"], cfg.eps)
    k = rope(k, positions, cfg.rope_base)
    v = (feature @ f64(lw["w_v"]).T).reshape(T, nkv, d)
    return k, v


def inject_context(cfg, W, target_hidden, positions):
    """Feature + per-layer injection for T new context tokens at ``positions``.

    Returns a list over layers of (K [T, nkv, d], V [T, nkv, d])."""
    f = context_feature(cfg, W, target_hidden)
    return [inject_layer(cfg, lw, f, positions) for lw in W["layers"]]


# --------------------------------------------------------------------------
# [DF2] "Arquitectura del Sistema" item 2: dynamic short convolution
# --------------------------------------------------------------------------
def short_conv(cfg, y, w_c, b_c) -> np.ndarray:
    """Two-tap depthwise dynamic convolution along the block ([DF2] item 2):
    one tap on the current position, one on the previous one; coefficients
    adapt to the current hidden state and every 16 channels share one
    correction; block-local and stateless (y_{-1} = 0).

    y: [S, H] -> [S, H];  [a; b] = tanh(W_c y_j + b_c) with a, b in R^{H/16}.
    """
    y = np.asarray(y, dtype=np.float64)
    S, H = y.shape
    G = H // 16
    coef = np.tanh(y @ f64(w_c).T + f64(b_c))        # [S, 2G]
    a = np.repeat(coef[:, :G], 16, axis=1)            # channel c -> group c // 16
    b = np.repeat(coef[:, G:], 16, axis=1)
    y_prev = np.vstack([np.zeros((1, H)), y[:-1]])
    return y + a * y + b * y_prev


# --------------------------------------------------------------------------
# block attention: [DF] §2.2 parallel block diffusion; mask semantics from
# [FD] "Metodologia" 1 (Ajuste de Atencion), Mecanismo
# --------------------------------------------------------------------------
def block_attention(cfg, q, k_ctx, v_ctx, k_blk, v_blk) -> np.ndarray:
    """Every block query attends to every injected context key and to all
    block keys (bidirectional inside the block, no other block present).

    q: [S, nq, d]; k_ctx, v_ctx: [n, nkv, d]; k_blk, v_blk: [S, nkv, d]
    -> [S, nq, d]."""
    keys = np.concatenate([np.asarray(k_ctx, np.float64).reshape(-1, cfg.n_kv_heads, cfg.head_dim), k_blk], 0)
    vals = np.concatenate([np.asarray(v_ctx, np.float64).reshape(-1, cfg.n_kv_heads, cfg.head_dim), v_blk], 0)
    S, nq, d = q.shape
    g = cfg.q_per_kv
    out = np.zeros((S, nq, d))
    for h in range(nq):
        kvh = h // g
        s = q[:, h, :] @ keys[:, kvh, :].T / np.sqrt(d)
        out[:, h, :] = softmax(s) @ vals[:, kvh, :]
    return out


# --------------------------------------------------------------------------
# drafter forward: [DF] §2.2 (parallel block diffusion), §2.3 (anchor,
# shared embedding and LM head), §3 item 1 (few layers)
# --------------------------------------------------------------------------
def drafter_forward(cfg, W, kv_ctx, n_ctx: int, anchor: int):
    """One forward pass of the drafter over a block of S = cfg.block positions
    (16, or a smaller runtime block size).

    Position 0 holds the clean anchor token ([DF] §2.3, anchor sampling
    mirrors inference), positions 1..S-1 the mask token; the block sits at
    absolute positions n_ctx .. n_ctx+S-1 after the injected context.
    kv_ctx: list over layers of (K [n_ctx, nkv, d], V [n_ctx, nkv, d]).

    Returns (h [S, H] final-normed hidden, z [S-1, V] logits of the mask
    positions from the shared LM head).
    """
    S, H = cfg.block, cfg.hidden
    nq, nkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    ids = [int(anchor)] + [cfg.mask_id] * (S - 1)
    pos = n_ctx + np.arange(S)
    x = f64(np.asarray(W["embed"])[ids])
    for l, lw in enumerate(W["layers"]):
        conv = lw.get("conv") if cfg.use_conv else None
        u = rms_norm(x, lw["g_attn"], cfg.eps)
        if conv:
            u = short_conv(cfg, u, *conv["pre_attn"])
        q = (u @ f64(lw["w_q"]).T).reshape(S, nq, d)
        k = (u @ f64(lw["w_k"]).T).reshape(S, nkv, d)
        v = (u @ f64(lw["w_v"]).T).reshape(S, nkv, d)
        if cfg.qk_norm:
            q = rms_norm(q, lw["g_q"], cfg.eps)
            k = rms_norm(k, lw["g_k"], cfg.eps)
        q = rope(q, pos, cfg.rope_base)
        k = rope(k, pos, cfg.rope_base)
        kc, vc = kv_ctx[l]
        o = block_attention(cfg, q, kc, vc, k, v).reshape(S, nq * d)
        a = o @ f64(lw["w_o"]).T
        if conv:
            a = short_conv(cfg, a, *conv["post_attn"])
        x = x + a
        u = rms_norm(x, lw["g_ffn"], cfg.eps)
        if conv:
            u = short_conv(cfg, u, *conv["pre_ffn"])
        m = (silu(u @ f64(lw["w_gate"]).T) * (u @ f64(lw["w_up"]).T)) @ f64(lw["w_down"]).T
        if conv:
            m = short_conv(cfg, m, *conv["post_ffn"])
        x = x + m
    h = rms_norm(x, W["g_final"], cfg.eps)
    z = h[1:] @ f64(W["lm_head"]).T
    return h, z


# --------------------------------------------------------------------------
# [DF2] "Arquitectura del Sistema" item 1: top-16 candidates and the Path
# Selector
# --------------------------------------------------------------------------
def top_k(z, k: int = 16):
    """Top-k per row by (value descending, token id ascending).
    z: [R, V] -> (ids [R, k] int32, values [R, k] float64)."""
    z = np.asarray(z, dtype=np.float64)
    R, V = z.shape
    ids = np.empty((R, k), dtype=np.int32)
    vals = np.empty((R, k), dtype=np.float64)
    tok = np.arange(V)
    for r in range(R):
        order = np.lexsort((tok, -z[r]))[:k]
        ids[r] = order
        vals[r] = z[r, order]
    return ids, vals


def context_gate(cfg, sel, h) -> np.ndarray:
    """Scalar context gate per mask position: sigmoid(w_g . h_j + b_g).
    h: [S, H] final-normed hidden -> [S-1]."""
    return sigmoid(np.asarray(h, np.float64)[1:] @ f64(sel["w_g"]) + float(sel["b_g"]))


def pair_scores(cfg, sel, anchor: int, cand_ids, cand_logits, h) -> np.ndarray:
    """Adjacent-pair scores s[j, p, c] for mask positions j = 1..J (J = S-1).

    score = drafter logit of candidate c + gate_j * (A e256[p]) . (B e256[c]),
    a low-rank bilinear compatibility on 256-d token embeddings under a
    context gate; p runs over the previous position's candidates (the anchor
    for the first mask position, repeated over the 16 rows).
    cand_ids, cand_logits: [J, 16] -> s: [J, 16, 16] indexed [j-1, p, c]."""
    cand_ids = np.asarray(cand_ids, dtype=np.int64)
    zc = np.asarray(cand_logits, dtype=np.float64)
    e = sel["e256"]
    A = f64(sel["a"])
    Bm = f64(sel["b"])
    gate = context_gate(cfg, sel, h)
    prev = np.vstack([np.full((1, cand_ids.shape[1]), int(anchor)), cand_ids[:-1]])
    up = f64(np.asarray(e)[prev]) @ A.T          # [J, 16, r]
    wc = f64(np.asarray(e)[cand_ids]) @ Bm.T     # [J, 16, r]
    bil = np.einsum("jpr,jcr->jpc", up, wc)
    return zc[:, None, :] + gate[:, None, None] * bil


def greedy_path(scores, cand_ids) -> np.ndarray:
    """Greedy traversal over precomputed pair scores: at each position take
    the best continuation of the previously chosen candidate (ties to the
    lower token id).  Returns draft ids [J]."""
    s = np.asarray(scores, dtype=np.float64)
    cand_ids = np.asarray(cand_ids)
    J, K, _ = s.shape
    path = np.empty(J, dtype=np.int32)
    p = 0
    for j in range(J):
        best = 0
        for c in range(1, K):
            if s[j, p, c] > s[j, p, best] or (s[j, p, c] == s[j, p, best]
                                               and cand_ids[j, c] < cand_ids[j, best]):
                best = c
        path[j] = cand_ids[j, best]
        p = best
    return path


def select_path(cfg, W, anchor, cand_ids, cand_logits, h):
    """DFlash-2 mode: pair scores + greedy path.  Otherwise (DFlash-1): the
    top-1 candidate per position.  Returns (draft [J], scores or None)."""
    cand_ids = np.asarray(cand_ids)
    if not cfg.use_selector:
        return cand_ids[:, 0].astype(np.int32), None
    s = pair_scores(cfg, W["sel"], anchor, cand_ids, cand_logits, h)
    return greedy_path(s, cand_ids), s


# --------------------------------------------------------------------------
# [DF2] "Flujo de Inferencia" steps 4-5 and [BW] "Contexto tecnico":
# greedy prefix verification
# --------------------------------------------------------------------------
def verify_greedy(draft, target):
    """Accept the longest prefix of the draft that equals the target's own
    tokens, then take the target's token at the first mismatch (the bonus);
    the rest is discarded.

    draft: [J]; target: [J+1] -> (k accepted drafts, bonus, committed [J+1]
    = target[0..k] followed by -1)."""
    draft = np.asarray(draft)
    target = np.asarray(target)
    n = draft.shape[0]
    k = 0
    while k < n and draft[k] == target[k]:
        k += 1
    committed = np.full(n + 1, -1, dtype=np.int32)
    committed[:k + 1] = target[:k + 1]
    return k, int(target[k]), committed


# --------------------------------------------------------------------------
# [DF2] "Arquitectura del Sistema" item 1: the other selection and
# verification modes - sampling over the precomputed pair scores, and
# rejection sampling that restores the target's exact distribution
# --------------------------------------------------------------------------
def inverse_cdf(weights, u: float) -> int:
    """Index of the first element whose running sum (in index order) exceeds
    u * total; the last positive weight when rounding leaves none."""
    w = np.asarray(weights, dtype=np.float64)
    total = w.sum()
    c = np.cumsum(w)
    hit = np.nonzero(c > u * total)[0]
    if hit.size:
        return int(hit[0])
    pos = np.nonzero(w > 0)[0]
    return int(pos[-1]) if pos.size else len(w) - 1


def sample_path(scores, cand_ids, temperature: float, uniforms):
    """Sampling over precomputed pair scores: at position j the draft
    distribution over the 16 candidates is q_j = softmax(s_j(c_{j-1}, .) / T)
    (c_0 = the anchor row), and c_j is drawn from it by inverse CDF in
    candidate order with the uniform u_j.  scores [J, 16, 16] (rows indexed
    by the previous candidate) -> (draft ids [J], q [J, 16], index [J])."""
    s = np.asarray(scores, dtype=np.float64)
    cand_ids = np.asarray(cand_ids)
    J, K, _ = s.shape
    draft = np.empty(J, dtype=np.int32)
    q = np.empty((J, K))
    idx = np.empty(J, dtype=np.int32)
    p = 0
    for j in range(J):
        row = s[j, p] / float(temperature)
        e = np.exp(row - row.max())
        q[j] = e / e.sum()
        c = inverse_cdf(q[j], float(uniforms[j]))
        draft[j], idx[j], p = cand_ids[j, c], c, c
    return draft, q, idx


def logit_scores(cand_logits) -> np.ndarray:
    """DFlash-1 (no selector): every previous candidate sees the drafter's
    own top-16 logits.  [J, 16] -> [J, 16, 16]."""
    z = np.asarray(cand_logits, dtype=np.float64)
    return np.repeat(z[:, None, :], z.shape[1], axis=1)


def verify_rejection(draft, q, cand_ids, target_logits, u_accept, u_bonus: float):
    """Rejection-sampling verification: draft token d_i (drawn from q_i) is
    accepted while u_i * q_i(d_i) < p_i(d_i), p_i = softmax of the target's
    logits at position i; at the first rejection the bonus is drawn from the
    residual max(0, p_i - q_i) (q_i zero outside the candidates), and after
    J acceptances from p_J; both by inverse CDF in vocabulary order with
    u_bonus.  The committed tokens then follow p exactly.
    target_logits [J+1, V] -> (k, bonus, committed [J+1], -1 padded)."""
    zt = np.asarray(target_logits, dtype=np.float64)
    draft = np.asarray(draft)
    cand_ids = np.asarray(cand_ids)
    q = np.asarray(q, dtype=np.float64)
    J = draft.shape[0]
    pt = np.exp(zt - zt.max(axis=1, keepdims=True))
    pt /= pt.sum(axis=1, keepdims=True)
    k = 0
    while k < J:
        c = int(np.nonzero(cand_ids[k] == draft[k])[0][0])
        if u_accept[k] * q[k, c] < pt[k, draft[k]]:
            k += 1
        else:
            break
    if k < J:
        r = pt[k].copy()
        r[cand_ids[k]] -= q[k]
        r = np.maximum(r, 0.0)
        bonus = inverse_cdf(r if r.sum() > 0 else pt[k], u_bonus)
    else:
        bonus = inverse_cdf(pt[J], u_bonus)
    committed = np.full(J + 1, -1, dtype=np.int32)
    committed[:k] = draft[:k]
    committed[k] = bonus
    return k, int(bonus), committed


# --------------------------------------------------------------------------
# one request end to end
# --------------------------------------------------------------------------
def draft_request(cfg, W, kv_ctx, n_ctx: int, anchor: int):
    """Draft one block for one request: forward, top-16, path selection.
    Returns a dict with h, z, cand_ids, cand_logits, draft, scores."""
    h, z = drafter_forward(cfg, W, kv_ctx, n_ctx, anchor)
    cand_ids, cand_logits = top_k(z, cfg.top_k)
    draft, scores = select_path(cfg, W, anchor, cand_ids, cand_logits, h)
    return {"h": h, "z": z, "cand_ids": cand_ids, "cand_logits": cand_logits,
            "draft": draft, "scores": scores}


def drafting_step(cfg, W, kv_ctx, n_ctx: int, new_hidden, anchor: int, target):
    """The steady-state step for one request: inject the new tokens' target
    features at positions n_ctx.., draft from the anchor after them, select a
    path, verify against ``target``.  kv_ctx is not modified."""
    T = 0 if new_hidden is None else np.asarray(new_hidden).shape[0]
    if T:
        new = inject_context(cfg, W, new_hidden, n_ctx + np.arange(T))
        kv = [(np.concatenate([np.asarray(k0, np.float64).reshape(-1, cfg.n_kv_heads, cfg.head_dim), k1]),
               np.concatenate([np.asarray(v0, np.float64).reshape(-1, cfg.n_kv_heads, cfg.head_dim), v1]))
              for (k0, v0), (k1, v1) in zip(kv_ctx, new)]
    else:
        kv = kv_ctx
    out = draft_request(cfg, W, kv, n_ctx + T, anchor)
    k, bonus, committed = verify_greedy(out["draft"], target)
    out.update(accept=k, bonus=bonus, committed=committed)
    return out
