"""Host-side weight packing on the CPU: the layouts include/dflash.h
documents (w_qkv = q, k, v rows; w_gu rows interleaved gate_i, up_i; FP8 row
scales packed exactly like their code rows) and the C structs that carry
the pointers.  Marshalling only, so it runs with CPU tensors."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from block_diffusion_drafter_context_gb300 import binding as B
from block_diffusion_drafter_context_gb300 import drafter as D
from synthetic import WORKLOADS, gen


def _np(t):
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _codes(a):
    return a.codes if hasattr(a, "codes") else np.asarray(a)


@pytest.mark.parametrize("name", ["T1", "T1F8", "T1D2F8"])
def test_packed_rows_follow_the_header(name):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    W = gen.make_weights(cfg, wl.seed)
    dw = D.upload_weights(cfg, W, device="cpu")
    fp8 = cfg.weight_fp8
    for lw, L in zip(W["layers"], dw["layers"]):
        q, k, v = (_codes(lw[n]) for n in ("w_q", "w_k", "w_v"))
        qkv = _np(L["w_qkv"])
        assert qkv.shape == (q.shape[0] + k.shape[0] + v.shape[0], cfg.hidden)
        assert np.array_equal(qkv, np.concatenate([q, k, v]))
        gate, up = _codes(lw["w_gate"]), _codes(lw["w_up"])
        gu = _np(L["w_gu"])
        assert gu.shape == (2 * cfg.ffn, cfg.hidden)
        assert np.array_equal(gu[0::2], gate) and np.array_equal(gu[1::2], up)
        if fp8:
            assert gu.dtype == np.uint8
            s_qkv = _np(L["s_qkv"])
            assert np.array_equal(s_qkv, np.concatenate([lw["w_q"].scale, lw["w_k"].scale, lw["w_v"].scale]))
            s_gu = _np(L["s_gu"])
            assert np.array_equal(s_gu[0::2], lw["w_gate"].scale) and np.array_equal(s_gu[1::2], lw["w_up"].scale)
            assert np.array_equal(_np(L["s_o"]), lw["w_o"].scale)
            assert np.array_equal(_np(L["s_down"]), lw["w_down"].scale)
            # every code row keeps its own scale: row r of the packed matrix
            # decodes to the source row it came from
            for packed_row, src, s_src in ((2 * 3 + 1, lw["w_up"], 3), (q.shape[0] + 2, lw["w_k"], 2)):
                codes = gu[packed_row] if src is lw["w_up"] else qkv[packed_row]
                scale = s_gu[packed_row] if src is lw["w_up"] else s_qkv[packed_row]
                assert np.array_equal(codes, src.codes[s_src]) and scale == src.scale[s_src]
        else:
            assert "s_qkv" not in L and gu.dtype == np.uint16
        if cfg.use_conv:
            assert len(L["w_conv"]) == 4 and len(L["b_conv"]) == 4
            G = cfg.hidden // 16
            for j, site in enumerate(D.CONV_SITES):
                # rows interleaved per channel group: 2g = current tap (row g
                # of [a; b]), 2g+1 = previous tap (row G + g)
                w_src, b_src = _codes(lw["conv"][site][0]), np.asarray(lw["conv"][site][1])
                w_pk, b_pk = _np(L["w_conv"][j]), _np(L["b_conv"][j])
                assert w_pk.shape == w_src.shape == (2 * G, cfg.hidden)
                assert np.array_equal(w_pk[0::2], w_src[:G]) and np.array_equal(w_pk[1::2], w_src[G:])
                assert np.array_equal(b_pk[0::2], b_src[:G]) and np.array_equal(b_pk[1::2], b_src[G:])
                if fp8:
                    s_src, s_pk = lw["conv"][site][0].scale, _np(L["s_conv"][j])
                    assert np.array_equal(s_pk[0::2], s_src[:G]) and np.array_equal(s_pk[1::2], s_src[G:])
    if fp8:
        assert np.array_equal(_np(dw["s_lm_head"]), W["lm_head"].scale)
        assert np.array_equal(_np(dw["lm_head"]), W["lm_head"].codes)


@pytest.mark.parametrize("name", ["T1F8", "T1D2"])
def test_weight_struct_points_at_the_packed_tensors(name):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    dw = D.upload_weights(cfg, gen.make_weights(cfg, wl.seed), device="cpu")
    w, lay = D.make_weights_struct(dw)
    for k in ("w_fc", "embed", "lm_head", "g_final"):
        assert getattr(w, k) == dw[k].data_ptr(), k
    assert bool(w.s_lm_head) == cfg.weight_fp8
    for i, L in enumerate(dw["layers"]):
        s = lay[i]
        for k in ("w_qkv", "w_o", "w_gu", "w_down", "g_attn", "g_ffn"):
            assert getattr(s, k) == L[k].data_ptr(), (i, k)
        if cfg.weight_fp8:
            assert s.s_gu == L["s_gu"].data_ptr() and s.s_qkv == L["s_qkv"].data_ptr()
        if cfg.use_conv:
            assert [s.w_conv[j] for j in range(4)] == [t.data_ptr() for t in L["w_conv"]]
    if cfg.use_selector:
        assert w.sel_e256 == dw["sel"]["e256"].data_ptr()
        assert w.sel_b_g == pytest.approx(dw["sel"]["b_g"])


def test_config_struct_carries_every_field():
    cfg = WORKLOADS["C3F8"].cfg
    c = D.make_config(cfg)
    assert c.dtype == B.DFLASH_BF16 and c.weight_fp8 == 1 and c.use_conv == 1 and c.use_selector == 1
    for k in ("hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "target_hidden",
              "n_target_layers", "sel_rank", "sel_dim", "page_size", "mask_id"):
        assert getattr(c, k) == getattr(cfg, k), k
    assert c.block_size == cfg.block and c.top_k == 16
    assert c.rope_base == pytest.approx(cfg.rope_base) and c.eps == pytest.approx(cfg.eps)


def test_paged_kv_templates_and_transposed_v():
    """A drawn cache state: pool page p of layer l holds template page
    page_map[l, p]; V pages are stored transposed ([d][slot])."""
    cfg = WORKLOADS["T1"].cfg
    rng = np.random.default_rng(5)
    L, T, nkv, P, d = cfg.n_layers, 3, cfg.n_kv_heads, cfg.page_size, cfg.head_dim
    tk = rng.standard_normal((L, T, nkv, P, d)).astype(np.float32)
    tv = rng.standard_normal((L, T, nkv, P, d)).astype(np.float32)
    num_pages = 5
    page_map = rng.integers(0, T, size=(L, num_pages))
    table = np.array([[0, 2, -1], [4, 1, 3]], dtype=np.int32)
    kv = D.PagedKV(cfg, table, num_pages, device="cpu")
    kv.fill_from_templates(tk, tv, page_map)
    k = kv.k.float().numpy()
    v = kv.v.float().numpy()
    bf = lambda a: torch.from_numpy(a).to(torch.bfloat16).float().numpy()   # noqa: E731
    for l in range(L):
        for p in range(num_pages):
            assert np.array_equal(k[l, p], bf(tk[l, page_map[l, p]]))
            assert np.array_equal(v[l, p], bf(tv[l, page_map[l, p]].transpose(0, 2, 1)))
    assert kv.max_pages == 3 and kv.struct.num_pages == num_pages
    assert kv.struct.k_cache == kv.k.data_ptr() and kv.struct.page_table == kv.page_table.data_ptr()
    r = kv.row(1)
    assert r.page_table == kv.page_table.data_ptr() + 3 * 4 and r.max_pages == 3
