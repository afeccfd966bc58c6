"""The allocation-free top-16 entry point against the existing one.

dflash_topk16_noalloc serves callers that cannot allocate device memory
(engine plugin hooks handed only their input and output buffers, under a
device-memory budget planned in advance): it keeps its scratch in a fixed
array inside the library.  Here it must reproduce the top-16 that
dflash_draft_block returns for the same logits, on two calls in a row (the
second call finds the first call's leftovers in the shared array).

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_noalloc_top16_matches_draft_block_twice():
    import torch

    from block_diffusion_drafter_context_gb300 import binding as Bd
    from block_diffusion_drafter_context_gb300.build import build
    from tests.gpu_case import Case

    build()
    c = Case("T1V")                      # vocab 40000: several chunks per row, so the scratch is used
    ref = c.draft(want_logits=True)
    torch.cuda.synchronize()
    rows, V = c.B * 15, c.cfg.vocab
    logits = ref["logits"].reshape(rows, V)
    for _ in range(2):
        ids = torch.full((rows, 16), -1, dtype=torch.int32, device="cuda")
        vals = torch.full((rows, 16), float("nan"), dtype=torch.float32, device="cuda")
        Bd.dflash_topk16_noalloc(logits, rows, V, ids, vals)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref["topk_ids"].reshape(rows, 16))
        assert torch.equal(vals, ref["topk_logits"].reshape(rows, 16))   # same values: tolerance 0
    # beyond the fixed limit: rejected, nothing launched
    with pytest.raises(Bd.DflashError) as e:
        Bd.dflash_topk16_noalloc(logits, 1025, V, ids, vals)
    assert e.value.code == -2


@pytest.mark.parametrize("rows,vocab", [(1024, 40001), (3, 151936)])
def test_noalloc_top16_matches_oracle_at_the_scratch_limits(rows, vocab):
    """Seeded N(0,1) fp32 logits against the oracle's top-16 (value
    descending, ties to the lower id) of the same values.  1024 rows is the
    row limit, and a vocabulary that is not a multiple of 4 takes the scalar
    load path; 3 rows of 151 936 fill all 32 chunks of the fixed scratch."""
    import torch

    import oracle as O
    from block_diffusion_drafter_context_gb300 import binding as Bd
    from block_diffusion_drafter_context_gb300.build import build

    build()
    z = np.random.default_rng(rows + vocab).standard_normal((rows, vocab), dtype=np.float32)
    ref_ids, ref_vals = O.top_k(z.astype(np.float64), 16)
    logits = torch.from_numpy(z).cuda()
    for _ in range(2):   # the second call finds the first call's leftovers in the shared array
        ids = torch.full((rows, 16), -1, dtype=torch.int32, device="cuda")
        vals = torch.full((rows, 16), float("nan"), dtype=torch.float32, device="cuda")
        Bd.dflash_topk16_noalloc(logits, rows, vocab, ids, vals)
        torch.cuda.synchronize()
        assert (ids.cpu().numpy() == ref_ids).all()
        assert (vals.cpu().numpy().astype(np.float64) == ref_vals).all()
