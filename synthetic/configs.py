"""Shapes and workload recipes for the synthetic DFlash drafting workloads.

This module holds sizes and seeds only: none of the drafting arithmetic lives
here.  Both the CUDA path (through its binding) and the fp64 oracle receive
the arrays that ``synthetic.gen`` builds from these recipes.

Workloads
---------
C0  tiny fp32 drafter, one request, 64 context tokens, seed 0.
C1  Qwen3-8B-shaped bf16 drafter, one request, 2048 context tokens.
C2  C1 shapes, 32 requests, ragged contexts uniform in [1024, 8192], 64-token
    KV pages, per-position match probability decaying 0.9 -> 0.5.
C3  C1 shapes plus the DFlash-2 pieces (dynamic short conv, Path Selector),
    8 requests, 4096 context tokens.
C4  27B-class drafter (hidden 5120, 40 q / 8 kv heads, FFN 17408), 64
    requests, ragged contexts uniform in [16384, 32768].  Its ~1.6 M context
    tokens start as a drawn cache state (template pages), not a prefill.
C1S5, C2S5  C1 and C2 run at a runtime block size of 5 (anchor + 4 mask
    positions), the engine-flag example of the DFlash-2 page; the drafter is
    unchanged (trained at 16, run at a smaller block).
C1F8, C2F8, C3F8  C1 / C2 / C3 with FP8 (E4M3, per-row scale) drafter
    weights: the "draft quantization" engine flag of the same page.

Small test-only workloads (``T*``) use ragged sizes (hidden 320, vocab 1000,
contexts that end mid-page, an empty context) so that every kernel sees
several tiles and a ragged tail while the oracle still finishes in seconds.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class DrafterConfig:
    name: str
    dtype: str              # "bf16" or "f32": storage and GEMM operand type
    hidden: int             # H
    n_layers: int           # L
    n_q_heads: int
    n_kv_heads: int
    head_dim: int           # d
    ffn: int                # F (SwiGLU width)
    vocab: int              # V (shared embedding / LM head rows)
    target_hidden: int      # H_t
    n_target_layers: int    # n_sel sampled target layers
    target_depth: int       # total target layers the n_sel are sampled from
    block: int = 16         # S (2..16): anchor + S-1 mask positions
    top_k: int = 16
    use_conv: bool = False  # DFlash-2 dynamic short convolution
    use_selector: bool = False  # DFlash-2 Path Selector
    sel_rank: int = 32      # r of the low-rank bilinear form
    sel_dim: int = 256      # width of the selector token embeddings
    qk_norm: bool = True
    fc_norm: bool = True
    # GPU precision mode: GEMM activations carried as bf16 high + low halves.
    # Needed where the DFlash-2 conv coefficients amplify bf16 rounding of the
    # activations past the 2% bound; plain bf16 activations elsewhere.
    split_act: bool = False
    # FP8 E4M3 GEMM weights with per-row fp32 scales (weight-only: the
    # activations stay bf16); the engine flag "draft quantization"
    weight_fp8: bool = False
    rope_base: float = 1e6
    eps: float = 1e-6
    page_size: int = 64

    @property
    def mask_id(self) -> int:
        return self.vocab - 1

    @property
    def q_per_kv(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def feat_in(self) -> int:
        return self.n_target_layers * self.target_hidden

    @property
    def conv_groups(self) -> int:
        return self.hidden // 16


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: DrafterConfig
    batch: int
    ctx_lo: int
    ctx_hi: int
    p_accept: tuple = field(default_factory=lambda: tuple([0.8] * 15))
    seed: int = 0
    explicit_ctx: tuple | None = None   # fixed context lengths (tests)
    # How the context KV is set up before the timed step: "inject" runs the
    # whole context through the injection projection; "template" draws the
    # cache state directly (seeded template pages mapped onto the pool), for
    # contexts whose target features would not fit in host memory.
    kv_fill: str = "inject"
    kv_templates: int = 256

    @property
    def ragged(self) -> bool:
        return self.explicit_ctx is not None or self.ctx_lo != self.ctx_hi


def _decay(p0: float, p1: float, n: int = 15) -> tuple:
    return tuple(p0 + (p1 - p0) * i / (n - 1) for i in range(n))


QWEN3_8B_SHAPED = DrafterConfig(
    name="qwen3-8b-shaped", dtype="bf16", hidden=4096, n_layers=5,
    n_q_heads=32, n_kv_heads=8, head_dim=128, ffn=12288, vocab=151936,
    target_hidden=4096, n_target_layers=5, target_depth=36)

TINY_F32 = DrafterConfig(
    name="tiny-f32", dtype="f32", hidden=256, n_layers=1,
    n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512, vocab=1024,
    target_hidden=256, n_target_layers=3, target_depth=12)

CLASS_27B = DrafterConfig(
    name="27b-class", dtype="bf16", hidden=5120, n_layers=5,
    n_q_heads=40, n_kv_heads=8, head_dim=128, ffn=17408, vocab=151936,
    target_hidden=5120, n_target_layers=5, target_depth=64)

# Ragged small bf16 drafter for parity tests: H=320 is 2.5 GEMM row tiles
# and not a multiple of the 64-wide K block; V=1000 is a ragged tile count.
SMALL_BF16 = DrafterConfig(
    name="small-bf16", dtype="bf16", hidden=320, n_layers=2,
    n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=704, vocab=1000,
    target_hidden=192, n_target_layers=3, target_depth=12)

WORKLOADS = {
    "C0": Workload("C0", TINY_F32, batch=1, ctx_lo=64, ctx_hi=64, seed=0),
    "C1": Workload("C1", QWEN3_8B_SHAPED, batch=1, ctx_lo=2048, ctx_hi=2048, seed=1),
    "C2": Workload("C2", QWEN3_8B_SHAPED, batch=32, ctx_lo=1024, ctx_hi=8192,
                   p_accept=_decay(0.9, 0.5), seed=2),
    "C3": Workload("C3", replace(QWEN3_8B_SHAPED, name="qwen3-8b-shaped-dflash2",
                                 use_conv=True, use_selector=True, split_act=True),
                   batch=8, ctx_lo=4096, ctx_hi=4096, seed=3),
    "C4": Workload("C4", CLASS_27B, batch=64, ctx_lo=16384, ctx_hi=32768, seed=4, kv_fill="template"),
    # FP8 drafter weights
    "C1F8": Workload("C1F8", replace(QWEN3_8B_SHAPED, name="qwen3-8b-shaped-fp8", weight_fp8=True),
                     batch=1, ctx_lo=2048, ctx_hi=2048, seed=1),
    "C2F8": Workload("C2F8", replace(QWEN3_8B_SHAPED, name="qwen3-8b-shaped-fp8", weight_fp8=True),
                     batch=32, ctx_lo=1024, ctx_hi=8192, p_accept=_decay(0.9, 0.5), seed=2),
    "C3F8": Workload("C3F8", replace(QWEN3_8B_SHAPED, name="qwen3-8b-shaped-dflash2-fp8", use_conv=True,
                                     use_selector=True, split_act=True, weight_fp8=True),
                     batch=8, ctx_lo=4096, ctx_hi=4096, seed=3),
    # runtime block size 5
    "C1S5": Workload("C1S5", replace(QWEN3_8B_SHAPED, name="qwen3-8b-shaped-block5", block=5),
                     batch=1, ctx_lo=2048, ctx_hi=2048, seed=1),
    "C2S5": Workload("C2S5", replace(QWEN3_8B_SHAPED, name="qwen3-8b-shaped-block5", block=5),
                     batch=32, ctx_lo=1024, ctx_hi=8192, p_accept=_decay(0.9, 0.5), seed=2),
    # test-only workloads
    "T0D2": Workload("T0D2", replace(TINY_F32, name="tiny-f32-dflash2",
                                     use_conv=True, use_selector=True),
                     batch=2, ctx_lo=0, ctx_hi=0, explicit_ctx=(64, 37), seed=10),
    "T1": Workload("T1", SMALL_BF16, batch=3, ctx_lo=0, ctx_hi=0,
                   explicit_ctx=(0, 100, 777), p_accept=_decay(0.9, 0.5), seed=11),
    "T1V": Workload("T1V", replace(SMALL_BF16, name="small-bf16-v40000", vocab=40000),
                    batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(7, 64, 129), seed=13),
    "T1D2": Workload("T1D2", replace(SMALL_BF16, name="small-bf16-dflash2",
                                     use_conv=True, use_selector=True, split_act=True),
                     batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(5, 64, 300), seed=12),
    # runtime block sizes below 16: 5 (bf16), 7 (fp32 DFlash-2), 2 (one mask position, bf16 DFlash-2)
    "T1S5": Workload("T1S5", replace(SMALL_BF16, name="small-bf16-block5", block=5),
                     batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(0, 63, 500), p_accept=_decay(0.9, 0.5), seed=14),
    "T0D2S7": Workload("T0D2S7", replace(TINY_F32, name="tiny-f32-dflash2-block7", use_conv=True,
                                         use_selector=True, block=7),
                       batch=2, ctx_lo=0, ctx_hi=0, explicit_ctx=(31, 90), seed=15),
    # FP8 weights: bf16 (every code planted in layer-0 W_q row 0 and LM-head
    # row 0) and DFlash-2 with split activations at block size 7
    "T1F8": Workload("T1F8", replace(SMALL_BF16, name="small-bf16-fp8", weight_fp8=True),
                     batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(0, 100, 777), p_accept=_decay(0.9, 0.5), seed=17),
    "T1D2F8": Workload("T1D2F8", replace(SMALL_BF16, name="small-bf16-dflash2-fp8", use_conv=True,
                                         use_selector=True, split_act=True, weight_fp8=True, block=7),
                       batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(5, 64, 300), seed=18),
    # 8 query heads per KV head (the attention's plain row layout) at block size 5
    "T1G8S5": Workload("T1G8S5", replace(SMALL_BF16, name="small-bf16-g8-block5", n_q_heads=8, n_kv_heads=1, block=5),
                       batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(10, 64, 450), seed=19),
    # one drafter layer (the context injection's single-group GEMM)
    "T1L1": Workload("T1L1", replace(SMALL_BF16, name="small-bf16-1layer", n_layers=1),
                     batch=2, ctx_lo=0, ctx_hi=0, explicit_ctx=(50, 130), seed=20),
    "T1D2S2": Workload("T1D2S2", replace(SMALL_BF16, name="small-bf16-dflash2-block2", use_conv=True,
                                         use_selector=True, split_act=True, block=2),
                       batch=3, ctx_lo=0, ctx_hi=0, explicit_ctx=(1, 64, 200), seed=16),
}

