"""ctypes binding of libdflash (include/dflash.h).

Argument marshalling only: every step of the drafting path runs in the CUDA
library.  The functions below carry the C names; tensors are passed as device
pointers (``tensor.data_ptr()``), streams as ``torch.cuda.Stream.cuda_stream``.
PyTorch is used for device memory and streams only.

If libdflash.so is missing the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char, c_double, c_float, c_int, c_size_t, c_ulonglong, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdflash.so")

DFLASH_BF16, DFLASH_F32 = 0, 1
ERR = {0: "OK", -1: "ARG", -2: "SHAPE", -3: "ALIGN", -4: "UNSUPPORTED", -5: "CUDA", -6: "TIMEOUT", -7: "DEVICE"}

# every entry point declared in include/dflash.h
EXPORTS = (
    "dflash_create", "dflash_destroy", "dflash_workspace_bytes", "dflash_inject_context",
    "dflash_draft_block", "dflash_select_path", "dflash_verify_greedy", "dflash_read_status",
    "dflash_set_wait_timeout", "dflash_set_gemm_ctas", "dflash_set_attn_split",
    "dflash_profile_begin", "dflash_profile_end", "dflash_debug_wait_flag", "dflash_last_error",
    "dflash_topk16_noalloc", "dflash_sample_path", "dflash_verify_rejection", "dflash_set_block_size",
    "dflash_get_block_size", "dflash_debug_e4m3_to_bf16", "dflash_debug_gemm_scratch_bytes", "dflash_debug_gemm",
    "dflash_debug_gemm_plan", "dflash_set_gemm_pairs", "dflash_fp8_weights_to_bf16",
    "dflash_debug_gemm_pair_clusters", "dflash_set_fused_topk",
)


class dflash_config(ctypes.Structure):
    _fields_ = [(n, c_int) for n in (
        "dtype", "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
        "target_hidden", "n_target_layers", "block_size", "top_k", "use_conv", "use_selector",
        "qk_norm", "fc_norm", "split_act", "sel_rank", "sel_dim", "mask_id", "page_size")] + [
        ("rope_base", c_float), ("eps", c_float), ("weight_fp8", c_int)]


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [("g_attn", c_void_p), ("w_qkv", c_void_p), ("g_q", c_void_p), ("g_k", c_void_p),
                ("w_o", c_void_p), ("g_ffn", c_void_p), ("w_gu", c_void_p), ("w_down", c_void_p),
                ("w_conv", c_void_p * 4), ("b_conv", c_void_p * 4),
                ("s_qkv", c_void_p), ("s_o", c_void_p), ("s_gu", c_void_p), ("s_down", c_void_p),
                ("s_conv", c_void_p * 4),
                ("w_qkv_bf16", c_void_p), ("w_o_bf16", c_void_p), ("w_gu_bf16", c_void_p), ("w_down_bf16", c_void_p),
                ("w_conv_bf16", c_void_p * 4)]


class dflash_weights(ctypes.Structure):
    _fields_ = [("w_fc", c_void_p), ("g_fc", c_void_p), ("embed", c_void_p), ("lm_head", c_void_p),
                ("g_final", c_void_p), ("layers", POINTER(dflash_layer_weights)),
                ("sel_e256", c_void_p), ("sel_a", c_void_p), ("sel_b", c_void_p),
                ("sel_w_g", c_void_p), ("sel_b_g", c_float), ("s_fc", c_void_p), ("s_lm_head", c_void_p),
                ("w_fc_bf16", c_void_p), ("lm_head_bf16", c_void_p)]


class dflash_kv(ctypes.Structure):
    _fields_ = [("k_cache", c_void_p), ("v_cache", c_void_p), ("page_table", c_void_p),
                ("num_pages", c_int), ("max_pages", c_int)]


class dflash_kernel_stat(ctypes.Structure):
    _fields_ = [("name", c_char * 32), ("launches", c_int), ("ms", c_double),
                ("bytes", c_double), ("flops", c_double)]


class DflashError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"dflash error {code} ({ERR.get(code, '?')}): {msg}")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load libdflash.so (raises if it was not built: no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    vp, i = c_void_p, c_int
    sig = {
        "dflash_create": (i, [POINTER(dflash_config), POINTER(dflash_weights), POINTER(c_void_p)]),
        "dflash_destroy": (None, [vp]),
        "dflash_workspace_bytes": (c_size_t, [vp, i, i]),
        "dflash_inject_context": (i, [vp, POINTER(dflash_kv), vp, vp, i, vp, vp, i, vp, c_size_t, vp]),
        "dflash_draft_block": (i, [vp, POINTER(dflash_kv), vp, vp, i, vp, vp, vp, vp, vp, c_size_t, vp]),
        "dflash_select_path": (i, [vp, vp, vp, vp, vp, i, vp, vp, vp, c_size_t, vp]),
        "dflash_verify_greedy": (i, [vp, vp, i, i, vp, vp, vp, vp]),
        "dflash_sample_path": (i, [vp, vp, vp, vp, vp, i, c_float, vp, vp, vp, vp, vp, c_size_t, vp]),
        "dflash_verify_rejection": (i, [vp, vp, vp, vp, vp, vp, vp, i, vp, vp, vp, vp, c_size_t, vp]),
        "dflash_read_status": (i, [vp, POINTER(c_int), vp]),
        "dflash_set_wait_timeout": (i, [vp, c_ulonglong]),
        "dflash_set_gemm_ctas": (i, [vp, i]),
        "dflash_set_gemm_pairs": (i, [vp, i]),
        "dflash_set_fused_topk": (i, [vp, i]),
        "dflash_set_attn_split": (i, [vp, i]),
        "dflash_set_block_size": (i, [vp, i]),
        "dflash_get_block_size": (i, [vp]),
        "dflash_profile_begin": (i, [vp]),
        "dflash_profile_end": (i, [vp, POINTER(dflash_kernel_stat), i, POINTER(c_int)]),
        "dflash_debug_wait_flag": (i, [vp, c_ulonglong, vp, vp]),
        "dflash_debug_e4m3_to_bf16": (i, [vp, i, vp, vp]),
        "dflash_fp8_weights_to_bf16": (i, [vp, i, i, vp, vp]),
        "dflash_debug_gemm_pair_clusters": (i, []),
        "dflash_debug_gemm_scratch_bytes": (c_size_t, []),
        "dflash_debug_gemm": (i, [vp, vp, i, vp, i, i, i, vp, vp, c_size_t, i, vp]),
        "dflash_debug_gemm_plan": (i, [i, i, i, i, i, i, i, i, i, i, vp]),
        "dflash_last_error": (ctypes.c_char_p, []),
        "dflash_topk16_noalloc": (i, [vp, i, i, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _p(x):
    """Device pointer of a tensor, an int, or None -> c_void_p."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _check(rc: int) -> int:
    if rc != 0:
        raise DflashError(rc, load().dflash_last_error().decode(errors="replace"))
    return rc


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return s if isinstance(s, int) else s.cuda_stream


# ---------------------------------------------------------------- C names
def dflash_create(cfg: dflash_config, w: dflash_weights) -> int:
    h = c_void_p()
    _check(load().dflash_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)))
    return h.value


def dflash_destroy(ctx: int) -> None:
    load().dflash_destroy(ctx)


def dflash_workspace_bytes(ctx: int, max_batch: int, max_new_tokens: int) -> int:
    return load().dflash_workspace_bytes(ctx, max_batch, max_new_tokens)


def dflash_inject_context(ctx, kv: dflash_kv, target_hidden, cu_new, total_new, ctx_len_in, ctx_len_out,
                          batch, workspace, workspace_bytes, stream=None):
    return _check(load().dflash_inject_context(ctx, ctypes.byref(kv), _p(target_hidden), _p(cu_new), total_new,
                                               _p(ctx_len_in), _p(ctx_len_out), batch, _p(workspace),
                                               workspace_bytes, _stream(stream)))


def dflash_draft_block(ctx, kv: dflash_kv, ctx_len, anchor_ids, batch, topk_ids, topk_logits, final_hidden,
                       logits, workspace, workspace_bytes, stream=None):
    return _check(load().dflash_draft_block(ctx, ctypes.byref(kv), _p(ctx_len), _p(anchor_ids), batch,
                                            _p(topk_ids), _p(topk_logits), _p(final_hidden), _p(logits),
                                            _p(workspace), workspace_bytes, _stream(stream)))


def dflash_select_path(ctx, anchor_ids, topk_ids, topk_logits, final_hidden, batch, draft_ids, pair_scores,
                       workspace, workspace_bytes, stream=None):
    return _check(load().dflash_select_path(ctx, _p(anchor_ids), _p(topk_ids), _p(topk_logits),
                                            _p(final_hidden), batch, _p(draft_ids), _p(pair_scores),
                                            _p(workspace), workspace_bytes, _stream(stream)))


def dflash_verify_greedy(draft_ids, target_ids, batch, block_size, accept_len, bonus, committed, stream=None):
    return _check(load().dflash_verify_greedy(_p(draft_ids), _p(target_ids), batch, block_size, _p(accept_len),
                                              _p(bonus), _p(committed), _stream(stream)))


def dflash_sample_path(ctx, anchor_ids, topk_ids, topk_logits, final_hidden, batch, temperature, uniforms,
                       draft_ids, draft_probs, pair_scores, workspace, workspace_bytes, stream=None):
    return _check(load().dflash_sample_path(ctx, _p(anchor_ids), _p(topk_ids), _p(topk_logits), _p(final_hidden),
                                            batch, float(temperature), _p(uniforms), _p(draft_ids),
                                            _p(draft_probs), _p(pair_scores), _p(workspace), workspace_bytes,
                                            _stream(stream)))


def dflash_verify_rejection(ctx, target_logits, draft_ids, topk_ids, draft_probs, u_accept, u_bonus, batch,
                            accept_len, bonus, committed, workspace, workspace_bytes, stream=None):
    return _check(load().dflash_verify_rejection(ctx, _p(target_logits), _p(draft_ids), _p(topk_ids),
                                                 _p(draft_probs), _p(u_accept), _p(u_bonus), batch,
                                                 _p(accept_len), _p(bonus), _p(committed), _p(workspace),
                                                 workspace_bytes, _stream(stream)))


def dflash_read_status(workspace, stream=None) -> int:
    """Returns the device status word (0 = clean) and clears it; never raises for it."""
    v = c_int(0)
    load().dflash_read_status(_p(workspace), ctypes.byref(v), _stream(stream))
    return v.value


def dflash_set_wait_timeout(ctx, ns: int):
    return _check(load().dflash_set_wait_timeout(ctx, ns))


def dflash_set_gemm_ctas(ctx, n: int):
    return _check(load().dflash_set_gemm_ctas(ctx, n))


def dflash_set_fused_topk(ctx, on: bool):
    return _check(load().dflash_set_fused_topk(ctx, int(bool(on))))


def dflash_set_gemm_pairs(ctx, on: bool):
    return _check(load().dflash_set_gemm_pairs(ctx, int(bool(on))))


def dflash_set_attn_split(ctx, tokens: int):
    return _check(load().dflash_set_attn_split(ctx, tokens))


def dflash_set_block_size(ctx, block_size: int):
    return _check(load().dflash_set_block_size(ctx, block_size))


def dflash_get_block_size(ctx) -> int:
    return int(load().dflash_get_block_size(ctx))


def dflash_debug_gemm_scratch_bytes() -> int:
    return int(load().dflash_debug_gemm_scratch_bytes())


def dflash_debug_gemm(W, w_scale, w_fp8, X, M, N, K, out, scratch, scratch_bytes, gemm_ctas=0, stream=None):
    return _check(load().dflash_debug_gemm(_p(W), _p(w_scale), int(w_fp8), _p(X), M, N, K, _p(out), _p(scratch),
                                           scratch_bytes, gemm_ctas, _stream(stream)))


GEMM_PLAN_KEYS = ("BN", "rtpg", "tok_tiles", "kbpt", "G", "csk", "tiles", "total", "partial_floats", "counters")


def dflash_debug_gemm_plan(M, N, K, n_groups=1, w_fp8=False, split_act=False, swiglu=False, per_sm=2, num_sms=152,
                           gemm_ctas=0) -> dict:
    out = (ctypes.c_longlong * len(GEMM_PLAN_KEYS))()
    _check(load().dflash_debug_gemm_plan(M, N, K, n_groups, int(w_fp8), int(split_act), int(swiglu), per_sm, num_sms,
                                         gemm_ctas, out))
    return dict(zip(GEMM_PLAN_KEYS, (int(v) for v in out)))


def dflash_debug_gemm_pair_clusters() -> int:
    return load().dflash_debug_gemm_pair_clusters()


def dflash_fp8_weights_to_bf16(codes, rows, cols, out, stream=None):
    return _check(load().dflash_fp8_weights_to_bf16(_p(codes), rows, cols, _p(out), _stream(stream)))


def dflash_debug_e4m3_to_bf16(codes, n, out, stream=None):
    return _check(load().dflash_debug_e4m3_to_bf16(_p(codes), n, _p(out), _stream(stream)))


def dflash_profile_begin(ctx):
    return _check(load().dflash_profile_begin(ctx))


def dflash_profile_end(ctx) -> list:
    n = c_int(0)
    buf = (dflash_kernel_stat * 64)()
    _check(load().dflash_profile_end(ctx, buf, 64, ctypes.byref(n)))
    return [{"name": buf[i].name.decode(), "launches": buf[i].launches, "ms": buf[i].ms,
             "bytes": buf[i].bytes, "flops": buf[i].flops} for i in range(min(n.value, 64))]


def dflash_debug_wait_flag(flag, timeout_ns: int, workspace, stream=None):
    return _check(load().dflash_debug_wait_flag(_p(flag), timeout_ns, _p(workspace), _stream(stream)))


def dflash_topk16_noalloc(logits, rows, vocab, topk_ids, topk_logits, stream=None):
    """Top-16 per row with the library's fixed scratch array (no device allocation)."""
    return _check(load().dflash_topk16_noalloc(_p(logits), rows, vocab, _p(topk_ids), _p(topk_logits),
                                               _stream(stream)))


def dflash_last_error() -> str:
    return load().dflash_last_error().decode(errors="replace")
