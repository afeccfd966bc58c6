"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on
the same seeded inputs.

Floats: max |err| <= 2e-2 * max |ref| (bf16) or 1e-4 (fp32) per tensor.
Integers: bit-exact, compared stage-isolated (the oracle's top-16 / path /
verify re-run on the GPU's own fp32 logits and hidden states), except where
the oracle's deciding gap is below 1e-3.
"""
import json
import os

import numpy as np
import pytest

import oracle as O
from synthetic import gen
from tests.gemm_cases import GEMM_EXACT_CASES
from tests.gpu_case import TOL, Case, rel_err, to_np

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_cases = {}


def case(name, **kw):
    key = (name, tuple(sorted(kw.items())))
    if key not in _cases:
        _cases[key] = Case(name, **kw)
    return _cases[key]


# ----------------------------------------------------------------- injection
@pytest.mark.parametrize("name", ["C0", "T0D2", "T1", "T1D2", "T1S5", "T1F8", "T1D2F8", "T1L1"])
def test_inject_matches_oracle(name):
    c = case(name)
    assert c.dr.status() == 0
    tol = TOL[c.cfg.dtype]
    assert to_np(c.ctx_d).tolist() == c.ctx.tolist()
    for b in range(c.B):
        if c.ctx[b] == 0:
            continue
        ref = c.oracle_kv(b)
        for l in range(c.cfg.n_layers):
            k, v = c.gpu_kv(b, l)
            assert rel_err(k, ref[l][0]) <= tol, (b, l, "K")
            assert rel_err(v, ref[l][1]) <= tol, (b, l, "V")


# ----------------------------------------------------------------- drafting
def _gap_ok(vals_sorted, i, thr=1e-3):
    """True if the value at rank i is separated from its neighbours by >= thr."""
    lo = vals_sorted[i] - vals_sorted[i + 1] if i + 1 < len(vals_sorted) else np.inf
    hi = vals_sorted[i - 1] - vals_sorted[i] if i > 0 else np.inf
    return min(lo, hi) >= thr


def end_to_end_ids(ids, z_gpu, z_ref):
    """Top-16 ids of one request against the oracle's own, end to end.

    Returns (checked, agree_1e3, ranks_1e3): `checked` asserts bit-exact ids
    at every rank whose oracle gap to both neighbours exceeds twice the
    measured max |logit error| (no rounding within that error can reorder
    them); the counts give the agreement rate under the 1e-3 gap rule."""
    err = float(np.abs(np.asarray(z_gpu, np.float64) - z_ref).max())
    oid = O.top_k(z_ref, 17)[0]
    full = -np.sort(-z_ref, axis=1)
    checked = agree = ranks = 0
    for j in range(z_ref.shape[0]):
        for r in range(16):
            if _gap_ok(full[j], r, 2 * err):
                assert ids[j, r] == oid[j, r], (j, r, err)
                checked += 1
            if _gap_ok(full[j], r):
                ranks += 1
                agree += int(ids[j, r] == oid[j, r])
    return checked, agree, ranks


@pytest.mark.parametrize("name", ["C0", "T0D2", "T1", "T1D2", "T1S5", "T0D2S7", "T1D2S2", "T1F8", "T1D2F8", "T1G8S5",
                                  "T1L1"])
def test_draft_matches_oracle(name):
    c = case(name)
    out = c.draft()
    assert c.dr.status() == 0
    tol = TOL[c.cfg.dtype]
    ids = to_np(out["topk_ids"])
    vals = to_np(out["topk_logits"])
    z = to_np(out["logits"])
    h = to_np(out["final_hidden"])
    for b in range(c.B):
        ref = c.oracle_draft(b)
        assert rel_err(h[b], ref["h"]) <= tol, (b, "final hidden")
        assert rel_err(z[b], ref["z"]) <= tol, (b, "logits")
        # stage-isolated: the oracle's top-16 of the GPU's own logits
        oid, oval = O.top_k(z[b].astype(np.float32).astype(np.float64), 16)
        assert (ids[b] == oid).all(), b
        assert (vals[b] == oval).all(), b
        # end to end: ids agree wherever the oracle's gap is decisive
        if c.cfg.dtype == "f32":
            full = -np.sort(-ref["z"], axis=1)
            for j in range(c.cfg.block - 1):
                for r in range(16):
                    if _gap_ok(full[j], r):
                        assert ids[b, j, r] == ref["cand_ids"][j, r], (b, j, r)
        else:
            checked, agree, ranks = end_to_end_ids(ids[b], z[b], ref["z"])
            print(f"{name} request {b}: end-to-end top-16 ids bit-exact at {checked} ranks beyond twice the logit "
                  f"error; {agree}/{ranks} agree where the oracle's gap is >= 1e-3")


@pytest.mark.parametrize("name,block", [("T1V", 5), ("T1S5", 5), ("T1D2F8", 7), ("T1D2S2", 2)])
def test_fused_top16_equals_logits_top16(name, block):
    """The LM head's top-16 epilogue (per-tile candidates + merge; taken when a
    call has at most 32 mask rows), with and without the logits written,
    against the logits + standalone top-16 and the oracle's top-16 of those
    logits: ids and values identical (vocabularies of 40 000 and 1 000, bf16
    and FP8 weights, split activations)."""
    from block_diffusion_drafter_context_gb300 import binding as Bd
    c = case(name)
    c.dr.set_block_size(block)
    assert c.B * (block - 1) <= 32
    Bd.dflash_set_fused_topk(c.dr.ctx, True)
    fused_nolog = c.draft(want_logits=False)
    fused = c.draft(want_logits=True)
    Bd.dflash_set_fused_topk(c.dr.ctx, False)
    plain = c.draft(want_logits=True)
    assert c.dr.status() == 0
    for out in (fused_nolog, fused):
        assert (to_np(out["topk_ids"]) == to_np(plain["topk_ids"])).all()
        assert (to_np(out["topk_logits"]) == to_np(plain["topk_logits"])).all()
    assert (to_np(fused["logits"]) == to_np(plain["logits"])).all()
    z = to_np(plain["logits"])
    for b in range(c.B):
        oid, oval = O.top_k(z[b], 16)
        assert (to_np(fused_nolog["topk_ids"])[b] == oid).all() and (to_np(fused_nolog["topk_logits"])[b] == oval).all()
    c.dr.set_block_size(c.cfg.block)


@pytest.mark.parametrize("name", ["T0D2", "T1D2", "T1", "T0D2S7", "T1D2S2", "T1D2F8"])
def test_select_path_matches_oracle(name):
    c = case(name)
    out = c.draft(want_logits=False)
    draft, scores = c.dr.select_path(c.anchor_d, out["topk_ids"], out["topk_logits"], out["final_hidden"])
    assert c.dr.status() == 0
    ids, vals, h = to_np(out["topk_ids"]), to_np(out["topk_logits"]), to_np(out["final_hidden"])
    draft = to_np(draft)
    for b in range(c.B):
        if not c.cfg.use_selector:
            assert (draft[b] == ids[b, :, 0]).all()
            continue
        s_ref = O.pair_scores(c.cfg, c.W["sel"], int(c.anchor[b]), ids[b], vals[b], h[b])
        s = to_np(scores)[b]
        assert rel_err(s, s_ref) <= 1e-4, b
        path_ref = O.greedy_path(s_ref, ids[b])
        p = 0
        for j in range(c.cfg.block - 1):
            row = np.sort(s_ref[j, p])[::-1]
            if row[0] - row[1] < 1e-3:
                break          # the oracle's own decision is within the gap: stop comparing
            assert draft[b, j] == path_ref[j], (b, j)
            p = int(np.where(ids[b, j] == path_ref[j])[0][0])


# ----------------------------------------------------------------- verification
def test_verify_golden_cases():
    import torch
    g = json.load(open(os.path.join(GOLDEN, "verify_cases.json")))["cases"]
    from block_diffusion_drafter_context_gb300.drafter import Drafter
    d = torch.tensor([c["draft"] for c in g], dtype=torch.int32, device="cuda")
    t = torch.tensor([c["target"] for c in g], dtype=torch.int32, device="cuda")
    acc, bonus, com = Drafter.verify_greedy(d, t)
    torch.cuda.synchronize()
    assert to_np(acc).tolist() == [c["k"] for c in g]
    assert to_np(bonus).tolist() == [c["bonus"] for c in g]
    assert to_np(com).tolist() == [c["committed"] for c in g]


def test_verify_golden_cases_short_blocks():
    import torch
    g = json.load(open(os.path.join(GOLDEN, "verify_cases_short_block.json")))["cases"]
    from block_diffusion_drafter_context_gb300.drafter import Drafter
    for S in sorted({c["S"] for c in g}):
        cs = [c for c in g if c["S"] == S]
        d = torch.tensor([c["draft"] for c in cs], dtype=torch.int32, device="cuda")
        t = torch.tensor([c["target"] for c in cs], dtype=torch.int32, device="cuda")
        acc, bonus, com = Drafter.verify_greedy(d, t)
        torch.cuda.synchronize()
        assert to_np(acc).tolist() == [c["k"] for c in cs]
        assert to_np(bonus).tolist() == [c["bonus"] for c in cs]
        assert to_np(com).tolist() == [c["committed"] for c in cs]


@pytest.mark.parametrize("S", [16, 5, 2])
def test_verify_random_against_oracle(S):
    import torch
    from block_diffusion_drafter_context_gb300.drafter import Drafter
    rng = np.random.default_rng(5)
    d = rng.integers(0, 50, size=(1000, S - 1)).astype(np.int32)
    t = gen.target_ids(d, [0.85] * 15, 50, seed=5)
    acc, bonus, com = Drafter.verify_greedy(torch.from_numpy(d).cuda(), torch.from_numpy(t).cuda())
    acc, bonus, com = to_np(acc), to_np(bonus), to_np(com)
    for b in range(1000):
        k, bo, cm = O.verify_greedy(d[b], t[b])
        assert (acc[b], bonus[b]) == (k, bo)
        assert (com[b] == cm).all()


# ----------------------------------------------------------------- the whole step
@pytest.mark.parametrize("name", ["T1", "T1D2", "T1S5", "T1D2S2", "T1F8"])
def test_step_is_lossless_and_verify_matches_oracle(name):
    import torch
    c = case(name)
    out = c.draft(want_logits=False)
    draft, _ = c.dr.select_path(c.anchor_d, out["topk_ids"], out["topk_logits"], out["final_hidden"])
    d = to_np(draft)
    t = gen.target_ids(d, c.wl.p_accept, c.cfg.vocab, seed=c.wl.seed)
    acc, bonus, com = c.dr.verify_greedy(draft, torch.from_numpy(t).cuda())
    acc, bonus, com = to_np(acc), to_np(bonus), to_np(com)
    for b in range(c.B):
        k, bo, cm = O.verify_greedy(d[b], t[b])
        assert (acc[b], bonus[b]) == (k, bo)
        assert (com[b] == cm).all()
        assert (com[b, :k + 1] == t[b, :k + 1]).all()


# ----------------------------------------------------------------- invariants
def test_stateless_isolated_and_cache_untouched():
    import torch
    c = case("T1")
    k0, v0 = c.kv.k.clone(), c.kv.v.clone()
    a = c.draft()
    b = c.draft()
    torch.cuda.synchronize()
    for key in ("topk_ids", "topk_logits", "final_hidden", "logits"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(k0, c.kv.k) and torch.equal(v0, c.kv.v)
    # perturb request 0 only: requests 1.. must not change at all
    anc = c.anchor_d.clone()
    anc[0] = (anc[0] + 7) % (c.cfg.vocab - 1)
    p = c.dr.draft_block(c.kv, c.ctx_d, anc, want_logits=True)
    torch.cuda.synchronize()
    assert not torch.equal(p["logits"][0], a["logits"][0])
    for key in ("topk_ids", "logits", "final_hidden"):
        assert torch.equal(p[key][1:], a[key][1:]), key


@pytest.mark.parametrize("name", ["T1", "T1F8"])
def test_single_request_views_match_oracle(name):
    """Each request drafted alone (batch 1 through a view of its page-table
    row: 16-token GEMM tiles, cluster split-K with pushed shares, cluster-mode
    attention) matches the oracle like the batched call does."""
    import types
    c = case(name)
    tol = TOL[c.cfg.dtype]
    for b in range(c.B):
        view = types.SimpleNamespace(struct=c.kv.row(b))
        out = c.dr.draft_block(view, c.ctx_d[b:b + 1], c.anchor_d[b:b + 1], want_logits=True)
        assert c.dr.status() == 0
        ref = c.oracle_draft(b)
        assert rel_err(to_np(out["final_hidden"])[0], ref["h"]) <= tol, b
        assert rel_err(to_np(out["logits"])[0], ref["z"]) <= tol, b


def test_runtime_block_size_switch_matches_oracle():
    """One context (configured block 16) switched between runtime block sizes
    from step to step: each step matches the oracle at that block size, and
    returning to 16 gives back the first step's results bit for bit."""
    from dataclasses import replace
    import torch
    c = case("T1")
    tol = TOL[c.cfg.dtype]
    first = c.draft()
    torch.cuda.synchronize()
    for S in (5, 2, 9):
        c.dr.set_block_size(S)
        out = c.draft()
        assert c.dr.status() == 0
        assert tuple(out["logits"].shape) == (c.B, S - 1, c.cfg.vocab)
        cfg_s = replace(c.cfg, block=S)
        for b in range(c.B):
            ref = O.draft_request(cfg_s, c.W, c.oracle_kv(b), int(c.ctx[b]), int(c.anchor[b]))
            assert rel_err(to_np(out["final_hidden"])[b], ref["h"]) <= tol, (S, b)
            assert rel_err(to_np(out["logits"])[b], ref["z"]) <= tol, (S, b)
    from block_diffusion_drafter_context_gb300.binding import DflashError
    with pytest.raises(DflashError):
        c.dr.set_block_size(17)
    c.dr.set_block_size(16)
    again = c.draft()
    torch.cuda.synchronize()
    for key in ("topk_ids", "topk_logits", "final_hidden", "logits"):
        assert torch.equal(first[key], again[key]), key


@pytest.mark.parametrize("name", ["T1", "T1F8"])
def test_split_kv_and_gemm_partition_do_not_change_results(name):
    import torch
    from block_diffusion_drafter_context_gb300 import binding as Bd
    c = case(name)
    ref = c.draft()
    ref_l = to_np(ref["logits"])
    for split in (64, 128, 256):
        Bd.dflash_set_attn_split(c.dr.ctx, split)
        out = c.draft()
        assert rel_err(to_np(out["logits"]), ref_l) <= 1e-2, split
    Bd.dflash_set_attn_split(c.dr.ctx, 0)
    for ctas in (1, 3, 7, 50):
        Bd.dflash_set_gemm_ctas(c.dr.ctx, ctas)
        out = c.draft()
        assert rel_err(to_np(out["logits"]), ref_l) <= 1e-2, ctas
    Bd.dflash_set_gemm_ctas(c.dr.ctx, 0)
    torch.cuda.synchronize()
    assert c.dr.status() == 0


def test_bounded_wait_reports_timeout_without_fault():
    import torch
    from block_diffusion_drafter_context_gb300 import binding as Bd
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    Bd.dflash_debug_wait_flag(flag, 200_000_000, ws)          # nothing ever sets the flag
    assert Bd.dflash_read_status(ws) == -6
    flag.fill_(1)
    Bd.dflash_debug_wait_flag(flag, 200_000_000, ws)
    assert Bd.dflash_read_status(ws) == 0
    torch.ones(1, device="cuda").sum().item()                 # context still usable


def test_e4m3_conversion_matches_oracle_decode_for_every_code():
    """The FP8 GEMM's code -> bf16 conversion over all 256 codes (the finite
    ones exactly, including the subnormals and both zeros) against the
    oracle's decode from the format definition."""
    import torch
    from block_diffusion_drafter_context_gb300 import binding as Bd
    codes = torch.arange(256, dtype=torch.uint8, device="cuda")
    out = torch.empty(256, dtype=torch.bfloat16, device="cuda")
    Bd.dflash_debug_e4m3_to_bf16(codes, 256, out)
    got = out.float().cpu().numpy().astype(np.float64)
    ref = O.e4m3_decode(np.arange(256))
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert (np.signbit(got[finite]) == np.signbit(ref[finite])).all()


def test_fp8_weight_bf16_copy_is_the_exact_decode():
    """dflash_fp8_weights_to_bf16 (the bf16 copies FP8 drafters keep for their
    tensor-bound launches): every finite code's value, exactly (the oracle's
    decode from the format definition), the row scales left apart."""
    import torch
    from block_diffusion_drafter_context_gb300 import binding as Bd
    rng = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    rows, cols = 37, 508
    codes = rng.choice(finite, size=(rows, cols)).astype(np.uint8)
    codes[0, :len(finite)] = finite
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    Bd.dflash_fp8_weights_to_bf16(torch.from_numpy(codes).cuda(), rows, cols, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = O.e4m3_decode(codes)
    assert np.array_equal(got, ref) and (np.signbit(got) == np.signbit(ref)).all()


# E4M3 codes of the integers 0..4 (1 = 0x38, 2 = 0x40, 3 = 0x44, 4 = 0x48); the sign bit negates
_E4M3_INT = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48}


@pytest.mark.parametrize("M,N,K,ctas,fp8", GEMM_EXACT_CASES)
def test_gemm_exact_on_small_integers(M, N, K, ctas, fp8):
    """The production GEMM (every decomposition: cluster split-K, one tile per
    CTA, stream-K with partial tiles; every token-tile width; bf16 and FP8
    weights) on integer inputs in [-4, 4]: every product and every fp32 sum
    is exact, so the result equals the integer matrix product bit for bit."""
    import torch
    from block_diffusion_drafter_context_gb300 import binding as Bd
    rng = np.random.default_rng(M * 7919 + N * 31 + K + ctas)
    Xi = rng.integers(-4, 5, size=(M, K))
    Wi = rng.integers(-4, 5, size=(N, K))
    X = torch.from_numpy(Xi.astype(np.float32)).to(torch.bfloat16).cuda()
    if fp8:
        codes = np.vectorize(lambda v: _E4M3_INT[abs(v)] | (0x80 if v < 0 else 0))(Wi).astype(np.uint8)
        W = torch.from_numpy(codes).cuda()
        sexp = rng.integers(-1, 2, size=N)                       # power-of-two row scales stay exact
        scale = torch.from_numpy((2.0 ** sexp).astype(np.float32)).cuda()
    else:
        W = torch.from_numpy(Wi.astype(np.float32)).to(torch.bfloat16).cuda()
        sexp, scale = np.zeros(N), None
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = Bd.dflash_debug_gemm_scratch_bytes()
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    Bd.dflash_debug_gemm(W, scale, fp8, X, M, N, K, out, scratch, nbytes, ctas)
    assert Bd.dflash_read_status(scratch) == 0
    ref = (Xi @ Wi.T).astype(np.float64) * (2.0 ** sexp)[None, :]
    assert np.array_equal(to_np(out), ref)
