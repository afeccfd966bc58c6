"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Every check here is independent of the oracle's own code path: closed forms,
invariants the method must have, hand-worked values (tests/golden), brute
force over tiny inputs, exhaustive enumeration of selector paths, and the
closed-form acceptance statistics of the synthetic target tokens.
"""
import itertools
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest

import oracle as O
from synthetic import gen
from synthetic.configs import TINY_F32, WORKLOADS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def micro_cfg(**kw):
    base = replace(TINY_F32, name="micro", hidden=32, n_layers=2, n_q_heads=4,
                   n_kv_heads=2, head_dim=8, ffn=48, vocab=40, target_hidden=16,
                   n_target_layers=3, rope_base=10000.0)
    return replace(base, **kw)


def f32_weights(cfg, seed=0):
    return gen.make_weights(cfg, seed)


def rand_kv(cfg, n, seed):
    r = np.random.default_rng(seed)
    return [(r.standard_normal((n, cfg.n_kv_heads, cfg.head_dim)),
             r.standard_normal((n, cfg.n_kv_heads, cfg.head_dim))) for _ in range(cfg.n_layers)]


# --------------------------------------------------------------------------
# storage decode
# --------------------------------------------------------------------------
def test_bf16_decode_exact():
    # 1.0 = 0x3F80, -2.5 = 0xC020, 0.15625 = 0x3E20
    bits = np.array([0x3F80, 0xC020, 0x3E20, 0x0000], dtype=np.uint16)
    assert O.f64(bits).tolist() == [1.0, -2.5, 0.15625, 0.0]


# --------------------------------------------------------------------------
# RMSNorm: closed forms
# --------------------------------------------------------------------------
def test_rms_norm_constant_vector_gives_gain():
    g = np.array([0.5, 1.5, -2.0, 3.0])
    for c in (1.0, 7.0, -3.0):
        y = O.rms_norm(np.full(4, c), g, 1e-6)
        np.testing.assert_allclose(y, np.sign(c) * g * abs(c) / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rms_norm_scale_invariant_and_unit_rms():
    r = np.random.default_rng(0)
    x = r.standard_normal((5, 64))
    y = O.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(37.0 * x, np.ones(64), 0.0), y, rtol=1e-13)


# --------------------------------------------------------------------------
# RoPE: hand-worked values, norm preservation, relative position
# --------------------------------------------------------------------------
def test_rope_golden_values():
    g = json.load(open(os.path.join(GOLDEN, "rope_example.json")))
    for c in g["cases"]:
        x = np.array(c["x"])[None, None, :]
        y = O.rope(x, np.array([c["pos"]]), g["base"])[0, 0]
        np.testing.assert_allclose(y, c["expected"], atol=1e-15)


def test_rope_preserves_norm_and_is_relative():
    r = np.random.default_rng(1)
    q = r.standard_normal((6, 3, 16))
    k = r.standard_normal((6, 3, 16))
    p = r.integers(0, 5000, 6)
    qr = O.rope(q, p, 1e6)
    np.testing.assert_allclose(np.linalg.norm(qr, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-13)
    for delta in (1, 1000, 77777):
        a = np.einsum("thd,shd->tsh", O.rope(q, p, 1e6), O.rope(k, p[::-1], 1e6))
        b = np.einsum("thd,shd->tsh", O.rope(q, p + delta, 1e6), O.rope(k, p[::-1] + delta, 1e6))
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)


# --------------------------------------------------------------------------
# attention: closed forms, brute force, mask invariants
# --------------------------------------------------------------------------
def test_attention_zero_query_is_mean_of_all_values():
    cfg = micro_cfg()
    r = np.random.default_rng(2)
    n = 23
    kc, vc = r.standard_normal((n, 2, 8)), r.standard_normal((n, 2, 8))
    kb, vb = r.standard_normal((16, 2, 8)), r.standard_normal((16, 2, 8))
    out = O.block_attention(cfg, np.zeros((16, 4, 8)), kc, vc, kb, vb)
    allv = np.concatenate([vc, vb])
    for h in range(4):
        np.testing.assert_allclose(out[:, h, :], np.broadcast_to(allv[:, h // 2].mean(0), (16, 8)), rtol=1e-13)


def test_attention_hand_worked_scale_and_head_grouping():
    """d = 8, scale 1/sqrt(8).  One context key k = e_0 on kv head 0 and
    sixteen zero block keys; query q = sqrt(8) ln 3 e_0.  Scores: ln 3 for the
    context key, 0 for the block keys -> weights 3/19 and 1/19 each.  With
    v_ctx = 19 e_0 and zero block values the output is 3 e_0, on query heads 0
    and 1 (both on kv head 0 with 2 query heads per kv head) and 0 on heads 2
    and 3 (kv head 1 holds zero keys and values).  A 1/d scale, no scale, or
    heads mapped h -> h mod nkv give other numbers."""
    cfg = micro_cfg()                     # 4 q heads, 2 kv heads, d = 8
    q = np.zeros((16, 4, 8))
    q[:, :, 0] = math.sqrt(8.0) * math.log(3.0)
    kc, vc = np.zeros((1, 2, 8)), np.zeros((1, 2, 8))
    kc[0, 0, 0] = 1.0
    vc[0, 0, 0] = 19.0
    out = O.block_attention(cfg, q, kc, vc, np.zeros((16, 2, 8)), np.zeros((16, 2, 8)))
    expect = np.zeros((16, 4, 8))
    expect[:, 0, 0] = expect[:, 1, 0] = 3.0
    np.testing.assert_allclose(out, expect, rtol=1e-13, atol=1e-13)


def test_attention_brute_force_loops():
    """Scalar-loop softmax attention over context + block, GQA head h -> h // g."""
    cfg = micro_cfg()
    r = np.random.default_rng(3)
    for n in (0, 5):
        q = r.standard_normal((16, 4, 8))
        kc, vc = r.standard_normal((n, 2, 8)), r.standard_normal((n, 2, 8))
        kb, vb = r.standard_normal((16, 2, 8)), r.standard_normal((16, 2, 8))
        out = O.block_attention(cfg, q, kc, vc, kb, vb)
        keys = list(kc) + list(kb)
        vals = list(vc) + list(vb)
        for i in range(16):
            for h in range(4):
                kv = h // 2
                sc = [sum(q[i, h, t] * kk[kv, t] for t in range(8)) / math.sqrt(8) for kk in keys]
                m = max(sc)
                w = [math.exp(s - m) for s in sc]
                tot = sum(w)
                ref = [sum(w[j] * vals[j][kv, t] for j in range(len(w))) / tot for t in range(8)]
                np.testing.assert_allclose(out[i, h], ref, rtol=1e-12, atol=1e-14)


def test_attention_mask_invariants():
    """In-block bidirectional, every context key visible (FlexDraft, Metodologia 1)."""
    cfg = micro_cfg()
    r = np.random.default_rng(4)
    n = 30
    q = r.standard_normal((16, 4, 8))
    kc, vc = r.standard_normal((n, 2, 8)), r.standard_normal((n, 2, 8))
    kb, vb = r.standard_normal((16, 2, 8)), r.standard_normal((16, 2, 8))
    base = O.block_attention(cfg, q, kc, vc, kb, vb)
    kb2, vb2 = kb.copy(), vb.copy()
    kb2[15] += 1.0
    vb2[15] += 1.0
    pert = O.block_attention(cfg, q, kc, vc, kb2, vb2)
    assert np.all(np.abs(pert[:15] - base[:15]).max(axis=(1, 2)) > 1e-6)   # not causal
    for t in (0, 17, 29):
        kc2, vc2 = kc.copy(), vc.copy()
        kc2[t] += 1.0
        vc2[t] -= 1.0
        p2 = O.block_attention(cfg, q, kc2, vc2, kb, vb)
        assert np.all(np.abs(p2 - base).max(axis=(1, 2)) > 1e-6)           # all context seen


def test_attention_context_order_irrelevant_and_gqa_equals_mha():
    cfg = micro_cfg()
    r = np.random.default_rng(5)
    n = 12
    q = r.standard_normal((16, 4, 8))
    kc, vc = r.standard_normal((n, 2, 8)), r.standard_normal((n, 2, 8))
    kb, vb = r.standard_normal((16, 2, 8)), r.standard_normal((16, 2, 8))
    base = O.block_attention(cfg, q, kc, vc, kb, vb)
    perm = r.permutation(n)
    np.testing.assert_allclose(O.block_attention(cfg, q, kc[perm], vc[perm], kb, vb), base, rtol=1e-12)
    mha = replace(cfg, n_kv_heads=4)
    rep = lambda a: np.repeat(a, 2, axis=1)
    np.testing.assert_allclose(O.block_attention(mha, q, rep(kc), rep(vc), rep(kb), rep(vb)), base, rtol=1e-12)


def test_attention_translation_invariant_through_injection():
    """K injected at absolute positions p and queried at p': shifting both by
    the same amount leaves the attention output unchanged."""
    cfg = micro_cfg(n_layers=1)
    W = f32_weights(cfg, 6)
    r = np.random.default_rng(6)
    X = r.standard_normal((20, cfg.feat_in))
    q = r.standard_normal((16, 4, 8))
    kb, vb = r.standard_normal((16, 2, 8)), r.standard_normal((16, 2, 8))
    outs = []
    for shift in (0, 4321):
        (k, v), = O.inject_context(cfg, W, X, np.arange(20) + shift)
        qq = O.rope(q, 20 + np.arange(16) + shift, cfg.rope_base)
        kk = O.rope(kb, 20 + np.arange(16) + shift, cfg.rope_base)
        outs.append(O.block_attention(cfg, qq, k, v, kk, vb))
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-9, atol=1e-11)


# --------------------------------------------------------------------------
# context feature and injection
# --------------------------------------------------------------------------
def test_context_feature_closed_forms():
    cfg = micro_cfg()
    W = f32_weights(cfg, 7)
    X = np.random.default_rng(7).standard_normal((9, cfg.feat_in))
    cfg0 = replace(cfg, eps=0.0)
    f = O.context_feature(cfg0, W, X)
    np.testing.assert_allclose(O.context_feature(cfg0, W, 3.5 * X), f, rtol=1e-12)
    g = O.f64(W["g_fc"])
    np.testing.assert_allclose(np.mean((f / g) ** 2, axis=-1), 1.0, rtol=1e-12)
    raw = O.context_feature(replace(cfg, fc_norm=False), W, X)
    np.testing.assert_allclose(raw, X @ O.f64(W["w_fc"]).T, rtol=1e-12)


def test_injected_k_has_unit_head_rms_before_rope():
    cfg = micro_cfg(n_layers=1)
    W = f32_weights(cfg, 8)
    X = np.random.default_rng(8).standard_normal((7, cfg.feat_in))
    (k, v), = O.inject_context(cfg, W, X, np.arange(7))
    g = O.f64(W["layers"][0]["g_k"])
    k0 = O.rope(k, -np.arange(7), cfg.rope_base)             # undo the rotation
    np.testing.assert_allclose(np.mean((k0 / g) ** 2, axis=-1), 1.0, rtol=1e-5)
    f = O.context_feature(cfg, W, X)
    np.testing.assert_allclose(v.reshape(7, -1), f @ O.f64(W["layers"][0]["w_v"]).T, rtol=1e-12)


# --------------------------------------------------------------------------
# dynamic short convolution
# --------------------------------------------------------------------------
def test_short_conv_golden_example():
    g = json.load(open(os.path.join(GOLDEN, "short_conv_example.json")))
    H = g["hidden"]
    cfg = micro_cfg(hidden=H)
    y = np.stack([np.arange(1, H + 1, dtype=float), 2.0 * np.arange(1, H + 1)])
    b_c = np.arctanh(np.array(g["tanh_targets"]["a"] + g["tanh_targets"]["b"]))
    out = O.short_conv(cfg, y, np.zeros((4, H)), b_c)
    np.testing.assert_allclose(out[0], g["expected"]["out0"], rtol=1e-12)
    np.testing.assert_allclose(out[1], g["expected"]["out1"], rtol=1e-12)


def test_short_conv_identity_locality_and_stateless():
    cfg = micro_cfg(hidden=64)
    r = np.random.default_rng(9)
    y = r.standard_normal((16, 64))
    np.testing.assert_array_equal(O.short_conv(cfg, y, np.zeros((8, 64)), np.zeros(8)), y)
    w, b = r.standard_normal((8, 64)) * 0.2, r.standard_normal(8)
    out = O.short_conv(cfg, y, w, b)
    # position 0 reads nothing before the block; position j reads only j, j-1
    y2 = y.copy()
    y2[5] += 1.0
    out2 = O.short_conv(cfg, y2, w, b)
    changed = np.abs(out2 - out).max(axis=1) > 0
    assert changed.tolist() == [j in (5, 6) for j in range(16)]
    # the block is stateless: position 0 equals a block that starts fresh there
    np.testing.assert_allclose(O.short_conv(cfg, y[3:], w, b)[0],
                               y[3] + np.repeat(np.tanh(y[3] @ w.T + b)[:4], 16) * y[3], rtol=1e-13)


# --------------------------------------------------------------------------
# top-k
# --------------------------------------------------------------------------
def test_top_k_matches_python_sort_with_ties():
    r = np.random.default_rng(10)
    z = np.round(r.standard_normal((6, 300)) * 3) / 2   # many exact ties
    z[2, :] = 0.0
    z[3, 7] = -0.0
    ids, vals = O.top_k(z, 16)
    for row in range(6):
        ref = sorted(range(300), key=lambda t: (-z[row, t], t))[:16]
        assert ids[row].tolist() == ref
        assert vals[row].tolist() == [z[row, t] for t in ref]


# --------------------------------------------------------------------------
# Path Selector: enumeration, special cases, brute-force scores
# --------------------------------------------------------------------------
def _sel_case(seed, J=15, K=16, V=50, E=6, r=3, H=8):
    rng = np.random.default_rng(seed)
    cfg = micro_cfg(hidden=H, vocab=V, sel_dim=E, sel_rank=r, use_selector=True)
    sel = {"e256": rng.standard_normal((V, E)), "a": rng.standard_normal((r, E)),
           "b": rng.standard_normal((r, E)), "w_g": rng.standard_normal(H), "b_g": 0.3}
    cand = np.stack([rng.permutation(V)[:K] for _ in range(J)])
    zc = -np.sort(-rng.standard_normal((J, K)), axis=1)
    h = rng.standard_normal((J + 1, H))
    anchor = int(rng.integers(V))
    return cfg, sel, anchor, cand, zc, h


def test_pair_scores_brute_force():
    cfg, sel, anchor, cand, zc, h = _sel_case(11, J=4, K=3)
    s = O.pair_scores(cfg, sel, anchor, cand, zc, h)
    e, A, B = sel["e256"], sel["a"], sel["b"]
    for j in range(4):
        gate = 1.0 / (1.0 + math.exp(-(sum(sel["w_g"][i] * h[j + 1, i] for i in range(cfg.hidden)) + sel["b_g"])))
        for p in range(3):
            tp = anchor if j == 0 else cand[j - 1, p]
            for c in range(3):
                tc = cand[j, c]
                bil = 0.0
                for rr in range(cfg.sel_rank):
                    up = sum(A[rr, i] * e[tp, i] for i in range(cfg.sel_dim))
                    wc = sum(B[rr, i] * e[tc, i] for i in range(cfg.sel_dim))
                    bil += up * wc
                assert s[j, p, c] == pytest.approx(zc[j, c] + gate * bil, rel=1e-12, abs=1e-12)


def test_pair_scores_hand_worked():
    """Rank 1, 2-wide embeddings: A picks coordinate 0 of the PREVIOUS token,
    B coordinate 1 of the CURRENT one, so u(p) . w(c) = e[p][0] * e[c][1].
    e[0] = (1, 0), e[1] = (0, 1), e[2] = (2, 3); zero logits; gate
    sigmoid(0) = 1/2 at position 1 and sigmoid(ln 3) = 3/4 at position 2.
    Position 1 (previous = anchor 2): s(c) = 1/2 * 2 * e[c][1] -> c = 0: 0,
    c = 1: 1, c = 2: 3.  Position 2, previous 2, current 1: 3/4 * 2 * 1 = 1.5;
    previous 0, current 2: 3/4 * 1 * 3 = 2.25; previous 1: 0 (e[1][0] = 0).
    Swapping A and B, or the gate's positions, changes these numbers."""
    cfg = micro_cfg(hidden=2, vocab=3, sel_dim=2, sel_rank=1, use_selector=True)
    sel = {"e256": np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 3.0]]), "a": np.array([[1.0, 0.0]]),
           "b": np.array([[0.0, 1.0]]), "w_g": np.array([1.0, 0.0]), "b_g": 0.0}
    h = np.array([[9.0, 9.0], [0.0, 5.0], [math.log(3.0), -5.0]])   # row 0 (the anchor) has no gate
    cand = np.array([[0, 1, 2], [0, 1, 2]])
    s = O.pair_scores(cfg, sel, 2, cand, np.zeros((2, 3)), h)
    assert s[0].tolist() == [[0.0, 1.0, 3.0]] * 3                   # every row: the anchor is the previous token
    assert s[1, 2, 1] == pytest.approx(1.5, abs=1e-15)
    assert s[1, 0, 2] == pytest.approx(2.25, abs=1e-15)
    assert s[1, 1].tolist() == [0.0, 0.0, 0.0]
    assert O.greedy_path(s, cand).tolist() == [2, 2]                # 3, then 3/4 * 2 * 3 = 4.5


@pytest.mark.parametrize("J", [1, 2, 3])
def test_greedy_path_against_exhaustive_enumeration(J):
    for seed in range(5):
        cfg, sel, anchor, cand, zc, h = _sel_case(100 + seed, J=J)
        s = O.pair_scores(cfg, sel, anchor, cand, zc, h)
        path = O.greedy_path(s, cand)
        idx = [int(np.where(cand[j] == path[j])[0][0]) for j in range(J)]
        # each greedy step is the argmax over the 16 continuations
        prev = 0
        for j in range(J):
            assert s[j, prev, idx[j]] == s[j, prev].max()
            prev = idx[j]
        # total of every one of the 16^J paths
        best = -np.inf
        for combo in itertools.product(range(16), repeat=J):
            tot, p = 0.0, 0
            for j, c in enumerate(combo):
                tot += s[j, p, c]
                p = c
            best = max(best, tot)
        greedy_tot = sum(s[j, ([0] + idx)[j], idx[j]] for j in range(J))
        assert greedy_tot <= best + 1e-12
        if J == 1:
            assert greedy_tot == best


def test_selector_special_cases_reduce_to_top1():
    cfg, sel, anchor, cand, zc, h = _sel_case(12)
    for mod in ("gate0", "a0"):
        s2 = dict(sel)
        if mod == "gate0":
            s2["w_g"] = np.zeros_like(sel["w_g"])
            s2["b_g"] = -700.0      # sigmoid ~ 1e-304
        else:
            s2["a"] = np.zeros_like(sel["a"])
        path = O.greedy_path(O.pair_scores(cfg, s2, anchor, cand, zc, h), cand)
        assert path.tolist() == cand[:, 0].tolist()


def test_selector_log_softmax_gives_same_path():
    cfg, sel, anchor, cand, zc, h = _sel_case(13)
    path = O.greedy_path(O.pair_scores(cfg, sel, anchor, cand, zc, h), cand)
    lse = np.log(np.exp(zc).sum(1, keepdims=True)) + 2.0
    path2 = O.greedy_path(O.pair_scores(cfg, sel, anchor, cand, zc - lse, h), cand)
    assert path.tolist() == path2.tolist()


# --------------------------------------------------------------------------
# verification
# --------------------------------------------------------------------------
def test_verify_golden_cases():
    g = json.load(open(os.path.join(GOLDEN, "verify_cases.json")))
    for c in g["cases"]:
        k, bonus, committed = O.verify_greedy(c["draft"], c["target"])
        assert (k, bonus, committed.tolist()) == (c["k"], c["bonus"], c["committed"]), c["name"]


def test_verify_golden_cases_short_blocks():
    g = json.load(open(os.path.join(GOLDEN, "verify_cases_short_block.json")))
    for c in g["cases"]:
        assert len(c["draft"]) == c["S"] - 1 and len(c["target"]) == c["S"]
        k, bonus, committed = O.verify_greedy(c["draft"], c["target"])
        assert (k, bonus, committed.tolist()) == (c["k"], c["bonus"], c["committed"]), c["name"]


@pytest.mark.parametrize("wl", ["C1", "C2"])
def test_acceptance_statistics_closed_form(wl):
    """E[k] = sum_i prod_{j<=i} p_j for the synthetic target tokens."""
    p = WORKLOADS[wl].p_accept
    closed, run = 0.0, 1.0
    for q in p:
        run *= q
        closed += run
    rng = np.random.default_rng(14)
    draft = rng.integers(0, 1000, size=(20000, 15))
    t = gen.target_ids(draft, p, 1000, seed=14)
    ks = np.array([O.verify_greedy(d, tt)[0] for d, tt in zip(draft, t)])
    assert abs(ks.mean() - closed) < 4 * ks.std() / math.sqrt(len(ks))
    assert {"C1": 3.859, "C2": 4.298}[wl] == pytest.approx(closed, abs=5e-4)


# --------------------------------------------------------------------------
# the whole drafter
# --------------------------------------------------------------------------
@pytest.mark.parametrize("S", [16, 5, 2])
def test_drafter_zero_sublayers_reduce_to_embedding_head(S):
    cfg = micro_cfg(block=S)
    W = f32_weights(cfg, 15)
    for lw in W["layers"]:
        lw["w_o"] = np.zeros_like(lw["w_o"])
        lw["w_down"] = np.zeros_like(lw["w_down"])
    anchor = 3
    h, z = O.drafter_forward(cfg, W, rand_kv(cfg, 10, 15), 10, anchor)
    assert h.shape == (S, cfg.hidden) and z.shape == (S - 1, cfg.vocab)
    e = O.f64(W["embed"])[[anchor] + [cfg.mask_id] * (S - 1)]
    hh = e / np.sqrt((e * e).mean(1, keepdims=True) + cfg.eps) * O.f64(W["g_final"])
    np.testing.assert_allclose(h, hh, rtol=1e-12)
    np.testing.assert_allclose(z, hh[1:] @ O.f64(W["lm_head"]).T, rtol=1e-12)


def test_drafter_hand_worked_swiglu_layer():
    """H = 2, one layer whose attention output projection is zero, so the
    anchor row is x = E[anchor] = (1, 1) plus the FFN.  Unit gains: the FFN
    input is (1, 1) (RMS 1).  Gate row 0 reads channel 0, up row 0 reads
    twice channel 1, down row 0 copies hidden unit 0:
    ffn = (silu(1) * 2, 0) = (1.462117, 0), x = (2.462117, 1), and the final
    RMSNorm gives h = x / sqrt((2.462117^2 + 1) / 2) = (1.310265, 0.532170).
    Gate and up swapped would give silu(2) * 1 = 1.761594 and h0 = 1.329719."""
    cfg = micro_cfg(hidden=2, n_layers=1, n_q_heads=1, n_kv_heads=1, ffn=2, vocab=5, target_hidden=2,
                    n_target_layers=1, block=2)
    W = f32_weights(cfg, 3)
    W["embed"] = np.ones((5, 2), np.float32)
    W["g_final"] = np.ones(2, np.float32)
    lw = W["layers"][0]
    lw["w_o"] = np.zeros_like(lw["w_o"])
    lw["g_ffn"] = np.ones(2, np.float32)
    lw["w_gate"] = np.array([[1, 0], [0, 0]], np.float32)
    lw["w_up"] = np.array([[0, 2], [0, 0]], np.float32)
    lw["w_down"] = np.array([[1, 0], [0, 0]], np.float32)
    h, _ = O.drafter_forward(cfg, W, rand_kv(cfg, 3, 3), 3, 0)
    np.testing.assert_allclose(h[0], [1.310265, 0.532170], atol=2e-6)
    np.testing.assert_allclose(h[1], h[0], rtol=1e-15)     # the mask row has the same embedding


def test_drafter_non_causal_all_context_and_stateless():
    cfg = micro_cfg()
    W = f32_weights(cfg, 16)
    kv = rand_kv(cfg, 20, 16)
    h, z = O.drafter_forward(cfg, W, kv, 20, 7)
    h_again, _ = O.drafter_forward(cfg, W, kv, 20, 7)
    np.testing.assert_array_equal(h, h_again)
    # the anchor position sees the later (mask) positions
    W2 = f32_weights(cfg, 16)
    W2["embed"] = W2["embed"].copy()
    W2["embed"][cfg.mask_id] += 0.5
    h2, _ = O.drafter_forward(cfg, W2, kv, 20, 7)
    assert np.abs(h2[0] - h[0]).max() > 1e-6
    # every context token reaches every position
    kv3 = [(k.copy(), v.copy()) for k, v in kv]
    kv3[0][1][13] += 1.0
    h3, _ = O.drafter_forward(cfg, W, kv3, 20, 7)
    assert np.all(np.abs(h3 - h).max(axis=1) > 1e-9)


def test_drafter_gqa_equals_duplicated_mha():
    cfg = micro_cfg()
    W = f32_weights(cfg, 17)
    kv = rand_kv(cfg, 9, 17)
    h, z = O.drafter_forward(cfg, W, kv, 9, 2)
    mha = replace(cfg, n_kv_heads=cfg.n_q_heads)
    W2 = f32_weights(cfg, 17)
    d = cfg.head_dim
    for lw in W2["layers"]:
        for nm in ("w_k", "w_v"):
            w = lw[nm].reshape(cfg.n_kv_heads, d, -1)
            lw[nm] = np.repeat(w, cfg.q_per_kv, axis=0).reshape(-1, cfg.hidden)
    kv2 = [(np.repeat(k, cfg.q_per_kv, axis=1), np.repeat(v, cfg.q_per_kv, axis=1)) for k, v in kv]
    h2, z2 = O.drafter_forward(mha, W2, kv2, 9, 2)
    np.testing.assert_allclose(h2, h, rtol=1e-12)
    np.testing.assert_allclose(z2, z, rtol=1e-11, atol=1e-12)


def test_zero_conv_dflash2_equals_dflash1_exactly():
    cfg1 = micro_cfg()
    cfg2 = micro_cfg(use_conv=True)
    W = f32_weights(cfg2, 18)
    for lw in W["layers"]:
        for s in lw["conv"]:
            w, b = lw["conv"][s]
            lw["conv"][s] = (np.zeros_like(w), np.zeros_like(b))
    kv = rand_kv(cfg1, 11, 18)
    h1, z1 = O.drafter_forward(cfg1, W, kv, 11, 5)
    h2, z2 = O.drafter_forward(cfg2, W, kv, 11, 5)
    np.testing.assert_array_equal(h1, h2)
    np.testing.assert_array_equal(z1, z2)


def test_drafting_step_is_lossless():
    """Committed tokens always equal the target's own continuation."""
    cfg = micro_cfg()
    W = f32_weights(cfg, 19)
    kv = rand_kv(cfg, 6, 19)
    rng = np.random.default_rng(19)
    for trial in range(4):
        X = rng.standard_normal((3, cfg.feat_in))
        out0 = O.draft_request(cfg, W, kv, 6, 1)
        t = gen.target_ids(out0["draft"][None], [0.7] * 15, cfg.vocab, seed=trial)[0]
        step = O.drafting_step(cfg, W, kv, 6, X, 1, t)
        k = step["accept"]
        assert step["committed"][:k + 1].tolist() == t[:k + 1].tolist()
        assert (step["committed"][k + 1:] == -1).all()
        assert step["bonus"] == t[k]


@pytest.mark.parametrize("S", [16, 5, 2])
def test_brute_force_micro_drafter_single_layer(S):
    """Scalar-loop transcription of one pre-norm layer + head on a micro
    drafter (1 layer, 2 q / 1 kv heads, d = 4), written from the layer
    reading, at the trained block size and at smaller runtime block sizes."""
    cfg = micro_cfg(hidden=8, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=4,
                    ffn=6, vocab=12, rope_base=10000.0, block=S)
    W = f32_weights(cfg, 20)
    n = 3
    kv = rand_kv(cfg, n, 20)
    anchor = 4
    h, z = O.drafter_forward(cfg, W, kv, n, anchor)
    F = lambda a: O.f64(a)
    lw = W["layers"][0]
    H, d = 8, 4

    def rms(v, g):
        ms = sum(t * t for t in v) / len(v)
        return [v[i] / math.sqrt(ms + cfg.eps) * float(g[i]) for i in range(len(v))]

    def mat(Wm, v):
        Wm = F(Wm)
        return [sum(Wm[o, i] * v[i] for i in range(len(v))) for o in range(Wm.shape[0])]

    def rot(v, p):
        out = list(v)
        for i in range(d // 2):
            th = p * cfg.rope_base ** (-2.0 * i / d)
            out[i] = v[i] * math.cos(th) - v[i + d // 2] * math.sin(th)
            out[i + d // 2] = v[i + d // 2] * math.cos(th) + v[i] * math.sin(th)
        return out

    E = F(W["embed"])
    x = [list(E[anchor if j == 0 else cfg.mask_id]) for j in range(S)]
    u = [rms(x[j], lw["g_attn"]) for j in range(S)]
    q = [[rot(rms(mat(lw["w_q"], u[j])[hh * d:(hh + 1) * d], lw["g_q"]), n + j) for hh in range(2)] for j in range(S)]
    k = [rot(rms(mat(lw["w_k"], u[j]), lw["g_k"]), n + j) for j in range(S)]
    v = [mat(lw["w_v"], u[j]) for j in range(S)]
    keys = [list(kv[0][0][t, 0]) for t in range(n)] + k
    vals = [list(kv[0][1][t, 0]) for t in range(n)] + v
    for j in range(S):
        o = []
        for hh in range(2):
            sc = [sum(q[j][hh][i] * kk[i] for i in range(d)) / math.sqrt(d) for kk in keys]
            m = max(sc)
            w = [math.exp(s - m) for s in sc]
            o += [sum(w[t] * vals[t][i] for t in range(len(w))) / sum(w) for i in range(d)]
        a = mat(lw["w_o"], o)
        x[j] = [x[j][i] + a[i] for i in range(H)]
        uf = rms(x[j], lw["g_ffn"])
        gt, up = mat(lw["w_gate"], uf), mat(lw["w_up"], uf)
        mid = [gt[i] / (1 + math.exp(-gt[i])) * up[i] for i in range(cfg.ffn)]
        mm = mat(lw["w_down"], mid)
        x[j] = [x[j][i] + mm[i] for i in range(H)]
    hb = [rms(x[j], W["g_final"]) for j in range(S)]
    np.testing.assert_allclose(h, hb, rtol=1e-11, atol=1e-12)
    zb = [mat(W["lm_head"], hb[j]) for j in range(1, S)]
    np.testing.assert_allclose(z, zb, rtol=1e-10, atol=1e-11)


# ------------------------------------------------------------------ sampling modes
def test_inverse_cdf_hand_worked():
    # running sums of [1, 2, 1] / 4 = 0.25, 0.75, 1.0: first one above u
    w = [1.0, 2.0, 1.0]
    assert O.inverse_cdf(w, 0.0) == 0
    assert O.inverse_cdf(w, 0.2499) == 0
    assert O.inverse_cdf(w, 0.25) == 1      # 0.25 is not above 0.25
    assert O.inverse_cdf(w, 0.7499) == 1
    assert O.inverse_cdf(w, 0.75) == 2
    assert O.inverse_cdf(w, 0.9999) == 2
    assert O.inverse_cdf([0.0, 3.0, 0.0], 0.5) == 1


def test_sample_path_low_temperature_is_greedy():
    rng = np.random.default_rng(21)
    for _ in range(20):
        s = rng.normal(size=(15, 16, 16))
        ids = np.stack([rng.permutation(1000)[:16] for _ in range(15)])
        d, q, idx = O.sample_path(s, ids, 1e-6, rng.random(15))
        assert (d == O.greedy_path(s, ids)).all()
        assert np.allclose(q.max(axis=1), 1.0)


def test_sample_path_frequencies_are_the_softmax():
    # one position: the share of a uniform grid that selects candidate c is q(c)
    rng = np.random.default_rng(22)
    s = rng.normal(size=(1, 16, 16)) * 2.0
    ids = np.arange(16)[None, :]
    T = 0.7
    grid = (np.arange(4000) + 0.5) / 4000
    counts = np.zeros(16)
    for u in grid:
        _, q, idx = O.sample_path(s, ids, T, [u])
        counts[idx[0]] += 1
    e = np.exp(s[0, 0] / T - (s[0, 0] / T).max())
    assert np.abs(counts / len(grid) - e / e.sum()).max() < 1e-3
    assert np.allclose(q[0], e / e.sum())


def test_sample_path_follows_the_previous_choice():
    # rows of the score table are indexed by the previous candidate
    s = np.zeros((2, 16, 16))
    s[0, 0, 5] = 50.0            # position 1 (from the anchor row) picks candidate 5
    s[1, 5, 9] = 50.0            # position 2 then reads row 5
    s[1, 0, 3] = 50.0            # a row it must not read
    ids = np.tile(np.arange(100, 116), (2, 1))
    d, _, idx = O.sample_path(s, ids, 1.0, [0.5, 0.5])
    assert idx.tolist() == [5, 9] and d.tolist() == [105, 109]


def test_rejection_sampling_is_lossless():
    # one position, V = 40: draft token drawn from q over 16 candidates, then
    # accept / residual.  Sweeping the accept uniform gives the acceptance
    # probability of each candidate; sweeping the bonus uniform after a
    # rejection gives the residual draw.  The first committed token must follow
    # the target distribution p exactly (to the grid's resolution).
    rng = np.random.default_rng(23)
    V = 40
    n = 2000
    grid = (np.arange(n) + 0.5) / n
    for trial in range(3):
        zt = rng.normal(size=(2, V)) * 1.5
        p = np.exp(zt[0] - zt[0].max())
        p /= p.sum()
        cand = rng.permutation(V)[:16]
        qv = rng.random(16) ** 3
        qv /= qv.sum()
        dist = np.zeros(V)
        for c in range(16):
            acc = np.mean([O.verify_rejection([cand[c]], qv[None, :], cand[None, :], zt, [ua], 0.0)[0] == 1
                           for ua in grid])
            dist[cand[c]] += qv[c] * acc
            if acc < 1.0:
                bon = np.zeros(V)
                for ub in grid:
                    bon[O.verify_rejection([cand[c]], qv[None, :], cand[None, :], zt, [1.0 - 1e-12], ub)[1]] += 1.0 / n
                dist += qv[c] * (1.0 - acc) * bon
        assert np.abs(dist - p).max() < 2e-3, (trial, np.abs(dist - p).max())


def test_rejection_special_cases():
    V = 30
    cand = np.arange(16)
    # the target puts all mass on the candidates and equals q there: always accept
    zt = np.full((16, V), -1e9)
    q = np.full((15, 16), 1.0 / 16)
    zt[:, :16] = 0.0
    draft = np.full(15, 3)
    for u in (0.0, 0.5, 0.999):
        k, bonus, com = O.verify_rejection(draft, q, np.tile(cand, (15, 1)), zt, np.full(15, u), 0.25)
        assert k == 15 and com[:15].tolist() == [3] * 15
        assert bonus == O.inverse_cdf(np.r_[np.ones(16), np.zeros(V - 16)], 0.25) == 4
    # the target gives the draft token no mass: reject at once, bonus from p minus q
    zt2 = np.zeros((16, V))
    zt2[0, 3] = -1e9
    k, bonus, com = O.verify_rejection(draft, q, np.tile(cand, (15, 1)), zt2, np.zeros(15), 0.0)
    assert k == 0 and bonus != 3 and com[1:].tolist() == [-1] * 15
    # residual max(0, p - q): tokens outside the candidates keep their full mass
    p0 = np.r_[np.zeros(1), np.ones(V - 1)] / (V - 1)
    r = np.maximum(p0 - np.r_[q[0], np.zeros(V - 16)], 0)
    assert bonus == O.inverse_cdf(r, 0.0) == 16


def test_logit_scores_ignore_the_previous_choice():
    z = np.random.default_rng(24).normal(size=(15, 16))
    s = O.logit_scores(z)
    assert s.shape == (15, 16, 16) and (s == z[:, None, :]).all()


# ------------------------------------------------------------------ FP8 drafter weights
def test_e4m3_decode_golden_values():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_values.json")))
    for c in g["cases"]:
        got = float(O.e4m3_decode(np.array([int(c["code"], 16)]))[0])
        if c["value"] == "nan":
            assert math.isnan(got), c["code"]
        else:
            assert got == c["value"] and math.copysign(1.0, got) == math.copysign(1.0, c["value"]), c["code"]


def test_e4m3_decode_structure():
    pos = O.e4m3_decode(np.arange(0x7F))
    assert (np.diff(pos) > 0).all()                       # codes 0x00..0x7E increase strictly
    assert pos[0] == 0.0 and pos[1] == 2.0 ** -9 and pos[-1] == 448.0
    # within one binade the step is the binade's 1/8; the subnormal step equals the first normal binade's
    assert np.allclose(np.diff(pos[:17]), 2.0 ** -9)
    neg = O.e4m3_decode(np.arange(0x80, 0xFF))
    np.testing.assert_array_equal(neg, -pos)              # the sign bit only negates


def test_fp8_quantizer_is_round_to_nearest_even():
    """The generator's per-row quantiser against brute force over the oracle's
    own decode table: every code is a nearest finite E4M3 value of w / scale,
    ties to the even code."""
    r = np.random.default_rng(40)
    w = np.concatenate([r.standard_normal((6, 200)) * 10 ** r.uniform(-4, 0, (6, 1)),
                        np.full((1, 200), 3.0)], 0).astype(np.float32)
    w[0, :5] = [0.0, -0.0, 1e-9, -1e-9, 448.0]
    q = gen.quantize_fp8_rows(w)
    table = O.e4m3_decode(np.arange(256))
    finite = np.array([c for c in range(256) if not np.isnan(table[c])])
    for n in range(w.shape[0]):
        assert q.scale[n] == np.float32(np.abs(w[n]).max() / np.float32(448.0))
        x = w[n].astype(np.float64) / float(q.scale[n])
        for k in range(w.shape[1]):
            d = np.abs(table[finite] - x[k])
            best = finite[d == d.min()]
            c = int(q.codes[n, k])
            assert c in best or (table[c] == 0.0 and (table[best] == 0.0).all()), (n, k, x[k], c)
            if len(best) > 1 and not (table[best] == 0.0).all():
                assert c % 2 == 0, (n, k)
    # a row's largest magnitude maps to +-448 exactly
    assert (np.abs(O.e4m3_decode(q.codes)).max(axis=1) == 448.0).all()


def test_fp8_planted_row_holds_every_finite_code():
    w = np.random.default_rng(41).standard_normal((3, 300)).astype(np.float32)
    q = gen.quantize_fp8_rows(w, plant_all_codes=True)
    codes = set(q.codes[0, :254].tolist())
    assert codes == {c for c in range(256) if (c & 0x7F) != 0x7F}


def test_brute_force_micro_dflash2_layer_with_short_convs():
    """Scalar-loop transcription of one DFlash-2 layer (the two-tap dynamic
    short convolution at its four sites: on the normed input and on the
    output of each sublayer, before the residual add; coefficients from the
    site's own input, one group per 16 channels, nothing before position 0),
    written from that reading, against the oracle's drafter forward."""
    S = 5
    cfg = micro_cfg(hidden=32, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=8,
                    ffn=20, vocab=12, rope_base=10000.0, block=S, use_conv=True)
    W = f32_weights(cfg, 21)
    n = 4
    kv = rand_kv(cfg, n, 21)
    anchor = 2
    h, z = O.drafter_forward(cfg, W, kv, n, anchor)
    F = lambda a: O.f64(a)
    lw = W["layers"][0]
    H, d, G = cfg.hidden, cfg.head_dim, cfg.hidden // 16

    def rms(v, g):
        ms = sum(t * t for t in v) / len(v)
        return [v[i] / math.sqrt(ms + cfg.eps) * float(g[i]) for i in range(len(v))]

    def mat(Wm, v):
        Wm = F(Wm)
        return [sum(Wm[o, i] * v[i] for i in range(len(v))) for o in range(Wm.shape[0])]

    def conv(site, rows):
        wc, bc = lw["conv"][site]
        out = []
        for j in range(S):
            c = [math.tanh(t + float(b)) for t, b in zip(mat(wc, rows[j]), F(bc))]
            prev = rows[j - 1] if j > 0 else [0.0] * H
            out.append([rows[j][ch] + c[ch // 16] * rows[j][ch] + c[G + ch // 16] * prev[ch] for ch in range(H)])
        return out

    def rot(v, p):
        out = list(v)
        for i in range(d // 2):
            th = p * cfg.rope_base ** (-2.0 * i / d)
            out[i] = v[i] * math.cos(th) - v[i + d // 2] * math.sin(th)
            out[i + d // 2] = v[i + d // 2] * math.cos(th) + v[i] * math.sin(th)
        return out

    E = F(W["embed"])
    x = [list(E[anchor if j == 0 else cfg.mask_id]) for j in range(S)]
    u = conv("pre_attn", [rms(x[j], lw["g_attn"]) for j in range(S)])
    q = [[rot(rms(mat(lw["w_q"], u[j])[hh * d:(hh + 1) * d], lw["g_q"]), n + j) for hh in range(2)] for j in range(S)]
    k = [rot(rms(mat(lw["w_k"], u[j]), lw["g_k"]), n + j) for j in range(S)]
    v = [mat(lw["w_v"], u[j]) for j in range(S)]
    keys = [list(kv[0][0][t, 0]) for t in range(n)] + k
    vals = [list(kv[0][1][t, 0]) for t in range(n)] + v
    att = []
    for j in range(S):
        o = []
        for hh in range(2):
            sc = [sum(q[j][hh][i] * kk[i] for i in range(d)) / math.sqrt(d) for kk in keys]
            m = max(sc)
            w = [math.exp(s - m) for s in sc]
            o += [sum(w[t] * vals[t][i] for t in range(len(w))) / sum(w) for i in range(d)]
        att.append(mat(lw["w_o"], o))
    att = conv("post_attn", att)
    x = [[x[j][i] + att[j][i] for i in range(H)] for j in range(S)]
    uf = conv("pre_ffn", [rms(x[j], lw["g_ffn"]) for j in range(S)])
    mm = []
    for j in range(S):
        gt, up = mat(lw["w_gate"], uf[j]), mat(lw["w_up"], uf[j])
        mm.append(mat(lw["w_down"], [gt[i] / (1 + math.exp(-gt[i])) * up[i] for i in range(cfg.ffn)]))
    mm = conv("post_ffn", mm)
    x = [[x[j][i] + mm[j][i] for i in range(H)] for j in range(S)]
    hb = [rms(x[j], W["g_final"]) for j in range(S)]
    np.testing.assert_allclose(h, hb, rtol=1e-10, atol=1e-12)
    zb = [mat(W["lm_head"], hb[j]) for j in range(1, S)]
    np.testing.assert_allclose(z, zb, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("S", [16, 5])
def test_incremental_injection_equals_one_shot(S):
    """A token's injected K/V depend only on its own feature and absolute
    position, so a steady-state step (inject T new tokens after n cached
    ones, then draft at n + T) equals injecting all n + T tokens at once and
    drafting after them.  Pins the positions the step uses."""
    cfg = micro_cfg(block=S)
    W = f32_weights(cfg, 22)
    r = np.random.default_rng(22)
    n, T = 9, S
    X = r.standard_normal((n + T, cfg.feat_in))
    kv_prefix = O.inject_context(cfg, W, X[:n], np.arange(n))
    target = np.zeros(S, dtype=np.int32)
    step = O.drafting_step(cfg, W, kv_prefix, n, X[n:], 3, target)
    kv_all = O.inject_context(cfg, W, X, np.arange(n + T))
    ref = O.draft_request(cfg, W, kv_all, n + T, 3)
    np.testing.assert_allclose(step["h"], ref["h"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(step["z"], ref["z"], rtol=1e-11, atol=1e-12)
    assert step["draft"].tolist() == ref["draft"].tolist()
    # and the positions matter: injecting the new tokens from position 0 changes the draft's inputs
    wrong = O.inject_context(cfg, W, X[n:], np.arange(T))
    kv_wrong = [(np.concatenate([k0, k1]), np.concatenate([v0, v1])) for (k0, v0), (k1, v1) in zip(kv_prefix, wrong)]
    bad = O.draft_request(cfg, W, kv_wrong, n + T, 3)
    assert np.abs(bad["h"] - ref["h"]).max() > 1e-6
