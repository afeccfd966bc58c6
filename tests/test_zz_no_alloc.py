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
