"""The seeded input recipe on the CPU: page tables are a permutation of the
pool with one run of pages per request, context lengths and anchors stay in
their ranges, synthetic target tokens differ from the draft exactly where
they reject it, and every generator is a pure function of its seed."""
import numpy as np
import pytest

from synthetic import WORKLOADS, gen


@pytest.mark.parametrize("name", ["T1", "C2", "C4"])
def test_page_table_is_a_permutation_of_the_pool(name):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    ctx = gen.context_lengths(wl)
    cap = ctx + cfg.block
    tab, total = gen.page_table(cap, cfg.page_size, wl.seed)
    need = (cap + cfg.page_size - 1) // cfg.page_size
    assert total == need.sum() and tab.shape == (wl.batch, need.max())
    used = np.concatenate([tab[b, :need[b]] for b in range(wl.batch)])
    assert np.array_equal(np.sort(used), np.arange(total))          # every page exactly once
    for b in range(wl.batch):
        assert (tab[b, need[b]:] == -1).all()
    tab2, _ = gen.page_table(cap, cfg.page_size, wl.seed)
    assert np.array_equal(tab, tab2)


def test_empty_and_single_token_requests_get_pages():
    tab, total = gen.page_table(np.array([0, 1, 64, 65]), 64, 3)
    assert total == 0 + 1 + 1 + 2
    assert (tab[0] == -1).all() and (tab[1, 1:] == -1).all() and (tab[3] >= 0).all()


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "T1"])
def test_context_lengths_and_anchors_in_range(name):
    wl = WORKLOADS[name]
    ctx = gen.context_lengths(wl)
    assert len(ctx) == wl.batch
    if wl.explicit_ctx is None:
        assert ctx.min() >= wl.ctx_lo and ctx.max() <= wl.ctx_hi
    a = gen.anchors(wl)
    assert a.min() >= 0 and a.max() <= wl.cfg.vocab - 2      # never the mask id V-1
    assert np.array_equal(a, gen.anchors(wl))                 # seeded
    if wl.batch > 4:
        assert not np.array_equal(a, gen.anchors(wl, step=1))   # a new draw per step


def test_target_ids_reject_exactly_where_they_differ():
    rng = np.random.default_rng(0)
    V, B, J = 50, 400, 15
    draft = rng.integers(0, V, size=(B, J))
    p = np.linspace(0.9, 0.5, J)
    t = gen.target_ids(draft, p, V, seed=11)
    assert t.shape == (B, J + 1) and t.min() >= 0 and t.max() < V
    match = t[:, :J] == draft
    # agreement rate per position follows p (binomial, 400 draws: within 5 sigma)
    rate = match.mean(0)
    assert (np.abs(rate - p) <= 5 * np.sqrt(p * (1 - p) / B)).all()
    # a rejected position never draws the draft token by accident
    t0 = gen.target_ids(draft, np.zeros(J), V, seed=11)
    assert (t0[:, :J] != draft).all()
    assert (gen.target_ids(draft, np.ones(J), V, seed=11)[:, :J] == draft).all()
    assert np.array_equal(t, gen.target_ids(draft, p, V, seed=11))


def test_normal_is_a_pure_function_of_seed_and_name():
    a = gen.normal((300, 70), 1.0, 5, "x")
    assert np.array_equal(a, gen.normal((300, 70), 1.0, 5, "x"))
    assert not np.array_equal(a, gen.normal((300, 70), 1.0, 5, "y"))
    assert not np.array_equal(a, gen.normal((300, 70), 1.0, 6, "x"))
    assert abs(a.mean()) < 0.05 and abs(a.std() - 1.0) < 0.05
    b = gen.normal((300, 70), 1.0, 5, "x", "bf16")
    assert b.dtype == np.uint16
    assert np.allclose(gen.bf16_bits_to_f32(b), a, rtol=2 ** -8, atol=0)
