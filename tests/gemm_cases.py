"""Shapes of the GEMM's bit-exact small-integer parity cases (M tokens, N
weight rows, K, forced stream-K CTAs (> 0), forced CTA pairs (< 0) or 0,
FP8 weights).  Shared by the GPU
test that runs them and the CPU test that checks, through the launch plan,
that they reach every decomposition and token tile."""

GEMM_EXACT_CASES = [
    (1, 448, 320, 0, False), (15, 4096, 1024, 0, False), (16, 1000, 4096, 0, False), (17, 448, 1024, 0, False),
    (33, 640, 1024, 0, False), (100, 1000, 320, 0, False), (300, 768, 1024, 0, False),
    (15, 4096, 1024, 5, False), (100, 1000, 1024, 7, False), (15, 24576, 512, 0, False),
    (15, 4096, 1024, 0, True), (17, 448, 1024, 0, True), (100, 1000, 320, 0, True), (300, 768, 1024, 0, True),
    (15, 4096, 1024, 5, True), (15, 24576, 512, 0, True),
    # several token tiles under stream-K, tiles split across CTAs
    (300, 768, 1024, 7, False), (300, 768, 1024, 7, True),
    # 256-token tiles on CTA pairs (2-SM MMA): one pair walking whole tiles,
    # pair tiles split across pairs (fixups), an odd row-tile count (the last
    # pair's phantom half), four token tiles, a 512-token projection
    (300, 768, 1024, -1, False), (300, 768, 1024, -5, False), (257, 896, 512, -3, False),
    (1024, 1152, 640, 0, False), (512, 4096, 4096, 0, False),
    # cluster split-K exchange with uneven row ranges (3 CTAs: 42 / 43 / 43
    # rows) and with 16 CTAs of 8 rows (a four-tile GEMM)
    (128, 6144, 4096, 0, False), (128, 512, 4096, 0, False),
]
