"""The tensor-core GEMM's launch decomposition, on the CPU (host arithmetic
only, through the library's plan hook; nothing is launched).

Expected plans for the drafter's projections are derived by hand from the
decomposition rules (token tile, cluster split-K for few tiles, one whole
tile per CTA between the SM count and the resident slots, stream-K
otherwise); the property test checks, over seeded random shapes, what every
plan must satisfy: the tiles cover the output, every CTA gets work, cluster
widths and CTA counts stay within their bounds, and the fp32 partial scratch
and tile counters a workspace holds always suffice."""
import random

import pytest

from block_diffusion_drafter_context_gb300 import binding as B
from block_diffusion_drafter_context_gb300 import build as BUILD
from synthetic import WORKLOADS

SMS = 152   # SMs of one GB300


@pytest.fixture(scope="module", autouse=True)
def lib():
    BUILD.build()
    return B.load()


def _shapes(cfg, tokens):
    """(name, M, N, K, groups, swiglu) of one drafting step's projections."""
    H, d = cfg.hidden, cfg.head_dim
    return {
        "fc": (tokens, H, cfg.n_target_layers * cfg.target_hidden, 1, False),
        "kv_inject": (tokens, cfg.n_kv_heads * d, H, 2 * cfg.n_layers, False),
        "qkv": (tokens, (cfg.n_q_heads + 2 * cfg.n_kv_heads) * d, H, 1, False),
        "o_proj": (tokens, H, cfg.n_q_heads * d, 1, False),
        "gate_up": (tokens, 2 * cfg.ffn, H, 1, True),
        "down": (tokens, H, cfg.ffn, 1, False),
        "lm_head": (tokens, cfg.vocab, H, 1, False),
    }


def _plan(M, N, K, groups, swiglu, f8=False, per_sm=2):
    return B.dflash_debug_gemm_plan(M, N, K, groups, f8, False, swiglu, per_sm, SMS)


# One request of 16 tokens, bf16 weights: 16-token tiles, two CTAs per SM
# (304 slots), at most 152 CTAs.
#   fc       32 tiles x 320 k-blocks: 64 <= 152 -> cluster split-K, min(8, 152/32, 320/8) = 4 -> 128 CTAs
#   kv_inject 10 groups x 8 tiles = 80: 160 > 152, 80 <= 152 -> stream-K, 5 120 iterations / 4 -> 152 CTAs
#   qkv      48 tiles: min(8, 152/48 = 3, 64/8) = 3 -> 144 CTAs
#   o_proj   32 tiles, 64 k-blocks: 4-way -> 128
#   gate_up  192 tiles: 152 < 192 <= 304 -> one whole tile per CTA, 192 CTAs
#   down     32 tiles, 192 k-blocks: 4-way -> 128
#   lm_head  1 187 tiles -> stream-K over 152 CTAs
C1_BF16 = {"fc": (128, 4), "kv_inject": (152, 1), "qkv": (144, 3), "o_proj": (128, 4), "gate_up": (192, 1),
           "down": (128, 4), "lm_head": (152, 1)}
# The same with FP8 weights: 128-code k-blocks, and the CTA cap is the 304
# slots (two MMA issuers per SM).
#   fc       32 tiles x 160: min(8, 304/32 = 9, 160/8 = 20) = 8 -> 256
#   kv_inject 80 tiles, 160 <= 304 -> cluster split-K: min(8, 3, max(2, 32/8 = 4)) = 3 -> 240
#   qkv      48 tiles x 32: min(8, 6, 4) = 4 -> 192
#   o_proj   32 x 32: min(8, 9, 4) = 4 -> 128
#   gate_up  192 tiles: 384 > 304, 152 < 192 <= 304 -> whole tiles, 192; SwiGLU: a power-of-two width anyway
#   down     32 x 96: min(8, 9, 12) = 8 -> 256
#   lm_head  1 187 tiles -> stream-K over 304 CTAs
C1_FP8 = {"fc": (256, 8), "kv_inject": (240, 3), "qkv": (192, 4), "o_proj": (128, 4), "gate_up": (192, 1),
          "down": (256, 8), "lm_head": (304, 1)}


@pytest.mark.parametrize("f8,expect", [(False, C1_BF16), (True, C1_FP8)], ids=["bf16", "fp8"])
def test_single_request_plans(f8, expect):
    cfg = WORKLOADS["C1"].cfg
    for name, (M, N, K, groups, swiglu) in _shapes(cfg, 16).items():
        p = _plan(M, N, K, groups, swiglu, f8=f8)
        assert p["BN"] == 16, name
        assert (p["G"], p["csk"]) == expect[name], name


def test_batched_plans_on_256_token_tiles():
    """32 requests (512 tokens), bf16: 256-token tiles, one CTA per SM.  fc,
    o_proj and down have 32 x 2 = 64 tiles (128 <= 152): 2-way cluster
    split-K; the rest stream-K with at most two pieces' partials per fixup
    (128 KB each), so at least 32 k-blocks per CTA: qkv 96 tiles x 64 =
    6 144 iterations / 32 -> 192, capped at 152."""
    cfg = WORKLOADS["C2"].cfg
    expect = {"fc": (128, 2), "o_proj": (128, 2), "down": (128, 2), "kv_inject": (152, 1), "qkv": (152, 1),
              "gate_up": (152, 1), "lm_head": (152, 1)}
    for name, (M, N, K, groups, swiglu) in _shapes(cfg, 32 * 16).items():
        p = _plan(M, N, K, groups, swiglu, per_sm=1)
        assert p["BN"] == 256 and p["tok_tiles"] == 2, name
        assert (p["G"], p["csk"]) == expect[name], name
    assert _plan(*_shapes(cfg, 512)["qkv"], per_sm=1)["total"] == 6144


def test_split_activations_and_fp8_cap_the_token_tile():
    for M, bn in ((1, 16), (16, 16), (17, 32), (33, 64), (65, 128), (128, 128), (129, 256), (5000, 256)):
        assert B.dflash_debug_gemm_plan(M, 4096, 4096)["BN"] == bn
        assert B.dflash_debug_gemm_plan(M, 4096, 4096, split_act=True)["BN"] == min(bn, 128)
        assert B.dflash_debug_gemm_plan(M, 4096, 4096, w_fp8=True)["BN"] == min(bn, 128)


def test_forced_cta_count_keeps_stream_k():
    for ctas in (1, 7, 152, 300, 100000):
        p = B.dflash_debug_gemm_plan(16, 6144, 4096, gemm_ctas=ctas)
        assert p["csk"] == 1 and p["G"] == min(ctas, p["total"] // 4)


def test_bad_arguments_are_rejected():
    for args in ((0, 1, 1), (1, 0, 1), (1, 1, 0), (-1, 1, 1)):
        with pytest.raises(B.DflashError):
            B.dflash_debug_gemm_plan(*args)
    with pytest.raises(B.DflashError):
        B.dflash_debug_gemm_plan(16, 128, 64, per_sm=0)
    with pytest.raises(B.DflashError):
        B.dflash_debug_gemm_plan(16, 128, 64, num_sms=0)


def _pieces_per_tile(p):
    """CTAs whose stream-K range [c*T/G, (c+1)*T/G) touches each tile."""
    T, G, kb = p["total"], p["G"], p["kbpt"]
    count = {}
    for c in range(G):
        b, e = c * T // G, (c + 1) * T // G
        if e > b:
            for t in range(b // kb, (e - 1) // kb + 1):
                count[t] = count.get(t, 0) + 1
    return count


def test_plan_properties_over_random_shapes():
    rng = random.Random(20261203)
    checked = 0
    for _ in range(3000):
        M = rng.choice([rng.randint(1, 1100), 16 * rng.randint(1, 64), rng.randint(1, 40)])
        groups = rng.choice([1, 1, 1, 2, 10, 16])
        N = 128 * rng.randint(1, 1200) if groups > 1 or rng.random() < 0.7 else rng.randint(1, 160000)
        f8 = rng.random() < 0.3
        K = 16 * rng.randint(1, 2000) if f8 else 8 * rng.randint(1, 4000)
        split = rng.random() < 0.3
        swiglu = rng.random() < 0.3
        sms = rng.choice([SMS, SMS, 148, 132, 20, 1])
        bn = B.dflash_debug_gemm_plan(M, N, K, groups, f8, split, swiglu, 1, sms)["BN"]
        # residency: two CTAs per SM only for token tiles up to 32 (larger
        # tiles take more than half an SM's shared memory)
        per_sm = rng.choice([1, 2]) if bn <= 32 else 1
        p = B.dflash_debug_gemm_plan(M, N, K, groups, f8, split, swiglu, per_sm, sms)
        BN, G, csk, tiles, kbpt = p["BN"], p["G"], p["csk"], p["tiles"], p["kbpt"]
        what = (M, N, K, groups, f8, split, swiglu, per_sm, sms)
        # the tiles cover the output exactly once
        assert (p["tok_tiles"] - 1) * BN < M <= p["tok_tiles"] * BN, what
        assert (p["rtpg"] - 1) * 128 < N <= p["rtpg"] * 128, what
        kstage = 128 if f8 else 64
        assert (kbpt - 1) * kstage < K <= kbpt * kstage, what
        assert tiles == p["rtpg"] * groups * p["tok_tiles"] and p["total"] == tiles * kbpt, what
        # every CTA gets at least one k-block
        assert 1 <= G <= p["total"], what
        slots = min(per_sm, 2) * sms
        cap = slots if f8 else sms
        if csk > 1:
            wide = 16 * tiles <= cap   # a handful of tiles: clusters up to the non-portable 16
            assert G == tiles * csk and csk <= min(16 if wide else 8, kbpt) and G <= cap and 2 * tiles <= cap, what
            if swiglu:
                assert csk & (csk - 1) == 0, what   # SwiGLU row pairs stay in one CTA
        else:
            assert G <= max(cap, tiles), what
            if sms < tiles <= slots:
                assert G == tiles, what             # one whole tile per CTA
            else:
                # stream-K: at least 4 k-blocks per CTA on average
                assert G <= max(1, -(-p["total"] // 4)), what
                # a fixup reads at most 256 KB of other pieces' fp32 partials
                pieces = max(_pieces_per_tile(p).values())
                assert (pieces - 1) * 128 * BN * 4 <= 256 * 1024, what
        # the workspace's scratch always suffices
        assert G * 2 * 128 * BN <= p["partial_floats"], what
        if tiles <= 4096:
            assert tiles <= p["counters"], what
        checked += 1
    assert checked == 3000


def test_exact_parity_cases_reach_every_decomposition():
    """The GPU's bit-exact GEMM cases, planned here as they are launched on
    one GB300: together they take cluster split-K, one whole tile per CTA and
    stream-K with tiles split across CTAs, with bf16 and with FP8 weights,
    and every bf16 token tile from 16 to 256."""
    from tests.gemm_cases import GEMM_EXACT_CASES
    seen = set()
    for M, N, K, ctas, f8 in GEMM_EXACT_CASES:
        if ctas < 0:   # forced CTA pairs: not a single-CTA plan
            continue
        bn = B.dflash_debug_gemm_plan(M, N, K, 1, f8, False, False, 1, SMS, ctas)["BN"]
        p = B.dflash_debug_gemm_plan(M, N, K, 1, f8, False, False, 2 if bn <= 32 else 1, SMS, ctas)
        if p["csk"] > 1:
            kind = "cluster"
        elif p["G"] == p["tiles"] and p["tiles"] > SMS:
            kind = "whole-tile"
        else:
            pieces = _pieces_per_tile(p)
            kind = "stream-k split" if max(pieces.values()) > 1 else "stream-k"
        seen.add((kind, f8))
        if not f8:
            seen.add(("BN", p["BN"]))
    for f8 in (False, True):
        for kind in ("cluster", "whole-tile", "stream-k split"):
            assert (kind, f8) in seen, (kind, f8)
    for bn in (16, 32, 64, 128, 256):
        assert ("BN", bn) in seen, bn
