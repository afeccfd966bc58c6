"""GPU parity of the sampling modes (path sampling over the scores,
rejection-sampling verification) against the fp64 oracle, stage-isolated on
the GPU's own candidates - on the small test workloads and on the full-size
C1 workload (vocabulary 151 936) - plus a distribution check of the GPU path.

Integer decisions are compared wherever the oracle's deciding margin is
decisive (> 1e-4 in probability); near a boundary the GPU's draw must still
be a valid one.  Random numbers are seeded inputs."""
import numpy as np
import pytest

import oracle as O
from tests.gpu_case import Case, to_np

pytestmark = pytest.mark.gpu

_cases = {}


def case(name):
    if name not in _cases:
        _cases[name] = Case(name)
    return _cases[name]


def cdf_margin(w, u):
    """Distance of u * total from the nearest running-sum boundary (fp64)."""
    w = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w) / w.sum()
    return float(np.min(np.abs(c - u)))


@pytest.mark.parametrize("name", ["T1", "T1D2", "T1S5", "T0D2S7", "C1"])
@pytest.mark.parametrize("temperature", [0.6, 1.0, 1.7])
def test_sample_path_matches_oracle(name, temperature):
    import torch
    c = case(name)
    J = c.cfg.block - 1
    out = c.draft(want_logits=False)
    rng = np.random.default_rng(31)
    u = rng.random((c.B, J)).astype(np.float32)
    draft, q = c.dr.sample_path(c.anchor_d, out["topk_ids"], out["topk_logits"], out["final_hidden"], temperature,
                                torch.from_numpy(u).cuda())
    assert c.dr.status() == 0
    ids, vals, h = to_np(out["topk_ids"]), to_np(out["topk_logits"]), to_np(out["final_hidden"])
    draft, q = to_np(draft), to_np(q)
    for b in range(c.B):
        s = (O.pair_scores(c.cfg, c.W["sel"], int(c.anchor[b]), ids[b], vals[b], h[b]) if c.cfg.use_selector
             else O.logit_scores(vals[b]))
        d_ref, q_ref, idx_ref = O.sample_path(s, ids[b], temperature, u[b].astype(np.float64))
        prev = 0
        for j in range(J):
            row = s[j, prev] / temperature
            e = np.exp(row - row.max())
            qj = e / e.sum()
            assert np.abs(q[b, j] - qj).max() < 1e-4, (b, j)
            if cdf_margin(qj, float(u[b, j])) < 1e-4:
                break          # the oracle's own draw is within rounding of a boundary: stop comparing
            assert draft[b, j] == d_ref[j], (b, j)
            prev = int(idx_ref[j])


def _target_logits(c, draft, rng, boost):
    """Synthetic target logits [B, S, V]: N(0, 1.5^2), the drafted token of
    each position raised by `boost` (so that acceptance varies)."""
    V, S = c.cfg.vocab, c.cfg.block
    z = rng.normal(size=(c.B, S, V)) * 1.5
    for b in range(c.B):
        for i in range(S - 1):
            z[b, i, draft[b, i]] += boost[i]
    return z.astype(np.float32)


@pytest.mark.parametrize("name", ["T1", "T1D2", "T1S5", "T1D2S2", "C1"])
def test_verify_rejection_matches_oracle(name):
    import torch
    c = case(name)
    J = c.cfg.block - 1
    out = c.draft(want_logits=False)
    rng = np.random.default_rng(32)
    checked = 0
    for trial in range(6):
        u = rng.random((c.B, J)).astype(np.float32)
        draft, q = c.dr.sample_path(c.anchor_d, out["topk_ids"], out["topk_logits"], out["final_hidden"], 1.0,
                                    torch.from_numpy(u).cuda())
        d, qn, ids = to_np(draft), to_np(q), to_np(out["topk_ids"])
        zt = _target_logits(c, d, rng, boost=np.linspace(6.0, 0.0, J) + trial)
        ua = rng.random((c.B, J)).astype(np.float32)
        ub = rng.random(c.B).astype(np.float32)
        acc, bonus, com = c.dr.verify_rejection(torch.from_numpy(zt).cuda(), draft, out["topk_ids"], q,
                                                torch.from_numpy(ua).cuda(), torch.from_numpy(ub).cuda())
        assert c.dr.status() == 0
        acc, bonus, com = to_np(acc), to_np(bonus), to_np(com)
        for b in range(c.B):
            z64 = zt[b].astype(np.float64)
            p = np.exp(z64 - z64.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            # accept decisions up to the oracle's first rejection, where decisive
            k_ref, bonus_ref, com_ref = O.verify_rejection(d[b], qn[b].astype(np.float64), ids[b], z64,
                                                           ua[b].astype(np.float64), float(ub[b]))
            margins = []
            for i in range(min(k_ref + 1, J)):
                cidx = int(np.nonzero(ids[b, i] == d[b, i])[0][0])
                margins.append(abs(float(ua[b, i]) * qn[b, i, cidx] - p[i, d[b, i]]))
            if min(margins) < 1e-5:
                continue
            assert acc[b] == k_ref, (trial, b)
            assert (com[b, :k_ref] == d[b, :k_ref]).all()
            # the bonus: a valid inverse-CDF draw, equal to the oracle's where decisive
            if k_ref < J:
                r = p[k_ref].copy()
                r[ids[b, k_ref]] -= qn[b, k_ref]
                w = np.maximum(r, 0.0)
            else:
                w = p[J]
            if cdf_margin(w, float(ub[b])) >= 1e-5:
                assert bonus[b] == bonus_ref, (trial, b)
            assert w[bonus[b]] > 0
            assert com[b, k_ref] == bonus[b] and (com[b, k_ref + 1:] == -1).all()
            checked += 1
    assert checked >= min(10, 3 * c.B)   # C1 (one request, full vocabulary): 6 trials


def test_rejection_output_follows_the_target_distribution():
    """2048 identical requests, independent uniforms: the first committed
    token's histogram matches p_0 within 4.5 standard errors per token."""
    import torch
    from block_diffusion_drafter_context_gb300.drafter import Drafter
    c = case("T1")
    n = 2048
    dr = Drafter(c.cfg, c.W, max_batch=n, max_new_tokens=16)
    rng = np.random.default_rng(33)
    V = c.cfg.vocab
    cand = rng.permutation(V)[:16].astype(np.int32)
    qv = rng.random(16) ** 2
    qv = (qv / qv.sum()).astype(np.float32)
    z0 = (rng.normal(size=V) * 1.2).astype(np.float32)
    z0[cand[:8]] += 2.5                      # the target overlaps the draft partly
    zt = np.broadcast_to(z0, (n, 16, V)).copy()
    ids = np.broadcast_to(cand, (n, 15, 16)).copy()
    q = np.broadcast_to(qv, (n, 15, 16)).copy()
    # each request's first draft token drawn from q by its own uniform
    ud = rng.random(n)
    first = np.array([cand[O.inverse_cdf(qv.astype(np.float64), x)] for x in ud], dtype=np.int32)
    draft = np.broadcast_to(cand[0], (n, 15)).copy()
    draft[:, 0] = first
    ua = rng.random((n, 15)).astype(np.float32)
    ub = rng.random(n).astype(np.float32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    acc, bonus, com = dr.verify_rejection(dev(zt), dev(draft), dev(ids), dev(q), dev(ua), dev(ub))
    torch.cuda.synchronize()
    assert dr.status() == 0
    com = to_np(com)
    p = np.exp(z0.astype(np.float64) - z0.max())
    p /= p.sum()
    hist = np.bincount(com[:, 0], minlength=V) / n
    se = np.sqrt(p * (1 - p) / n) + 1.0 / n
    assert (np.abs(hist - p) <= 4.5 * se).all(), np.abs(hist - p).max()
    dr.close()
