"""The C-ABI library loads, exports every entry point include/dflash.h
declares, its ctypes structs match the C layout, and host-side validation
rejects bad arguments - all without a GPU (no compute calls)."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from block_diffusion_drafter_context_gb300 import binding as B
from block_diffusion_drafter_context_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.load()


def declared_entry_points():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]*?\b(dflash_\w+)\s*\(", src)))


def test_header_declares_the_four_hot_path_calls():
    names = declared_entry_points()
    for n in ("dflash_inject_context", "dflash_draft_block", "dflash_select_path", "dflash_verify_greedy"):
        assert n in names
    assert sorted(B.EXPORTS) == names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_entry_points():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (dflash_\w+)", out))
    assert exported == set(declared_entry_points())


def test_struct_layouts_match_the_header():
    probe = r"""
#include <stdio.h>
#include <stddef.h>
#include "dflash.h"
#define P(T) printf(#T " %zu\n", sizeof(T));
#define O(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  P(dflash_config) P(dflash_layer_weights) P(dflash_weights) P(dflash_kv) P(dflash_kernel_stat)
  O(dflash_config, rope_base) O(dflash_config, eps) O(dflash_config, page_size) O(dflash_config, split_act)
  O(dflash_layer_weights, w_conv) O(dflash_layer_weights, b_conv)
  O(dflash_weights, layers) O(dflash_weights, sel_b_g) O(dflash_kv, num_pages) O(dflash_kernel_stat, ms)
  O(dflash_config, weight_fp8) O(dflash_layer_weights, s_qkv) O(dflash_layer_weights, s_conv)
  O(dflash_weights, s_fc) O(dflash_weights, s_lm_head)
  O(dflash_layer_weights, w_qkv_bf16) O(dflash_layer_weights, w_conv_bf16) O(dflash_weights, lm_head_bf16)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "p.c")
        open(c, "w").write(probe)
        exe = os.path.join(d, "p")
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.split() for l in lines if l)
    py = {
        "dflash_config": ctypes.sizeof(B.dflash_config),
        "dflash_layer_weights": ctypes.sizeof(B.dflash_layer_weights),
        "dflash_weights": ctypes.sizeof(B.dflash_weights),
        "dflash_kv": ctypes.sizeof(B.dflash_kv),
        "dflash_kernel_stat": ctypes.sizeof(B.dflash_kernel_stat),
        "dflash_config.rope_base": B.dflash_config.rope_base.offset,
        "dflash_config.eps": B.dflash_config.eps.offset,
        "dflash_config.page_size": B.dflash_config.page_size.offset,
        "dflash_config.split_act": B.dflash_config.split_act.offset,
        "dflash_layer_weights.w_conv": B.dflash_layer_weights.w_conv.offset,
        "dflash_layer_weights.b_conv": B.dflash_layer_weights.b_conv.offset,
        "dflash_weights.layers": B.dflash_weights.layers.offset,
        "dflash_weights.sel_b_g": B.dflash_weights.sel_b_g.offset,
        "dflash_kv.num_pages": B.dflash_kv.num_pages.offset,
        "dflash_kernel_stat.ms": B.dflash_kernel_stat.ms.offset,
        "dflash_config.weight_fp8": B.dflash_config.weight_fp8.offset,
        "dflash_layer_weights.s_qkv": B.dflash_layer_weights.s_qkv.offset,
        "dflash_layer_weights.s_conv": B.dflash_layer_weights.s_conv.offset,
        "dflash_weights.s_fc": B.dflash_weights.s_fc.offset,
        "dflash_weights.s_lm_head": B.dflash_weights.s_lm_head.offset,
        "dflash_layer_weights.w_qkv_bf16": B.dflash_layer_weights.w_qkv_bf16.offset,
        "dflash_layer_weights.w_conv_bf16": B.dflash_layer_weights.w_conv_bf16.offset,
        "dflash_weights.lm_head_bf16": B.dflash_weights.lm_head_bf16.offset,
    }
    for k, v in py.items():
        assert int(got[k]) == v, k


def _cfg(**kw):
    c = B.dflash_config()
    base = dict(dtype=0, hidden=256, n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=128, ffn=512, vocab=1024,
                target_hidden=256, n_target_layers=3, block_size=16, top_k=16, use_conv=0, use_selector=0,
                qk_norm=1, fc_norm=1, split_act=1, sel_rank=32, sel_dim=256, mask_id=1023, page_size=64, rope_base=1e6, eps=1e-6)
    base.update(kw)
    for k, v in base.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,code", [
    (dict(block_size=17), -4), (dict(block_size=1), -4), (dict(block_size=8), -3),   # 2..16 pass to the weights
    (dict(top_k=8), -4), (dict(page_size=32), -4), (dict(hidden=250), -2),
    (dict(n_kv_heads=3), -2), (dict(head_dim=96), -4), (dict(mask_id=5000), -1), (dict(dtype=7), -1),
    (dict(use_selector=1, sel_rank=100), -4),
    (dict(weight_fp8=1, dtype=1), -4),                 # FP8 weights: bf16 path only
    (dict(weight_fp8=1, ffn=520), -2),                 # FP8 code rows must be 16-byte multiples
])
def test_create_rejects_bad_configs_without_touching_the_gpu(lib, kw, code):
    w = B.dflash_weights()
    h = ctypes.c_void_p()
    rc = lib.dflash_create(ctypes.byref(_cfg(**kw)), ctypes.byref(w), ctypes.byref(h))
    assert rc == code
    assert h.value is None
    assert lib.dflash_last_error()


def test_create_rejects_missing_or_misaligned_weights(lib):
    w = B.dflash_weights()
    h = ctypes.c_void_p()
    assert lib.dflash_create(ctypes.byref(_cfg()), ctypes.byref(w), ctypes.byref(h)) == -3
    w.w_fc = w.embed = w.lm_head = w.g_final = 0x1008      # not 16-byte aligned
    assert lib.dflash_create(ctypes.byref(_cfg()), ctypes.byref(w), ctypes.byref(h)) == -3


def test_null_and_empty_calls(lib):
    assert lib.dflash_workspace_bytes(None, 1, 1) == 0
    assert lib.dflash_verify_greedy(None, None, 0, 16, None, None, None, None) == 0     # empty batch: no-op
    assert lib.dflash_verify_greedy(None, None, 3, 16, None, None, None, None) == -1
    assert lib.dflash_verify_greedy(None, None, 3, 17, None, None, None, None) == -1    # block size above 16
    assert lib.dflash_verify_greedy(None, None, 3, 1, None, None, None, None) == -1     # no mask position
    assert lib.dflash_draft_block(None, None, None, None, 1, None, None, None, None, None, 0, None) == -1
    assert lib.dflash_set_attn_split(None, 64) == -1
    assert lib.dflash_set_block_size(None, 5) == -1
    assert lib.dflash_debug_gemm(None, None, 0, None, 16, 128, 64, None, None, 0, 0, None) == -1
    assert lib.dflash_get_block_size(None) == 0


def test_noalloc_top16_validates_before_touching_the_device(lib):
    fake = 0x10000   # never dereferenced: every case below returns before any device work
    assert lib.dflash_topk16_noalloc(None, 0, 1000, None, None, None) == 0          # empty: no-op
    assert lib.dflash_topk16_noalloc(fake, -1, 1000, fake, fake, None) == -1
    assert lib.dflash_topk16_noalloc(None, 4, 1000, fake, fake, None) == -1
    assert lib.dflash_topk16_noalloc(fake, 1025, 1000, fake, fake, None) == -2      # over the fixed scratch
    assert "1024" in lib.dflash_last_error().decode()


def test_sampling_calls_reject_a_null_context(lib):
    assert lib.dflash_sample_path(None, None, None, None, None, 1, 1.0, None, None, None, None, None, 0, None) == -1
    assert lib.dflash_verify_rejection(None, None, None, None, None, None, None, 1, None, None, None, None, 0,
                                       None) == -1
    assert lib.dflash_select_path(None, None, None, None, None, 1, None, None, None, 0, None) == -1
    assert lib.dflash_inject_context(None, None, None, None, 16, None, None, 1, None, 0, None) == -1
