"""The launch planner on the host alone (fgemm_plan_on: no GPU is touched): which path runs, the
persistent grid, the tiles and how the last round is cut, the narrowed last column of tiles and
the ring / second-operand staging.  Every expected value is derived in a comment from the rules
stated in include/fgemm.h (fgemm_opts, fgemm_plan_info); the device is described as this GB300
(152 SMs, 76 CTA pairs resident)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import gemm_epilogue_gb300.binding as fg  # noqa: E402

SMS, PAIRS = 152, 76
# Device addresses that are never dereferenced: 16-byte aligned and far apart.
A, B, BIAS, Y, OUT = (0x10000000 + i * 0x10000000 for i in range(5))


def plan(M, N, K, dtype, gate=False, opts=None, sms=SMS, pairs=PAIRS, epilogue=None, a=A):
    return fg.fgemm_plan_on(a, B, BIAS, Y if gate or epilogue == fg.EPI_RESIDUAL_RELU else None,
                            OUT, M, N, K, dtype, sms, pairs, gate=gate, opts=opts,
                            epilogue=epilogue)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fg.lib()


def test_square_4096_on_cta_pairs():
    p = plan(4096, 4096, 4096, fg.BF16)
    # M > 128 and K > 512: CTA pairs, 256 x 256 tiles -> 16 x 16 = 256 tiles on 76 pairs
    assert (p["path"], p["cluster"], p["grid"], p["tiles"]) == (fg.PATH_TC, 2, 152, 256)
    # 256 = 3 x 76 + 28: the 28 tiles of the last round are cut in two (pairs: at most 2 pieces,
    # and 2 x 28 <= 76), so 228 + 56 = 284 work items
    assert (p["tail_split"], p["work_items"]) == (2, 284)
    # N a multiple of 256: the last column is full width; two K rows per stage on pairs
    assert (p["last_tile_n"], p["k_rows"], p["row_barriers"], p["resident_pairs"]) == (256, 2, 0, 76)


def test_gate_glu_block_k4096():
    p = plan(1024, 21568, 4096, fg.F16, gate=True)
    # 4 x 85 = 340 tiles; 340 = 4 x 76 + 36 -> 36 tiles in 2 pieces: 304 + 72 = 376 items
    assert (p["cluster"], p["tiles"], p["tail_split"], p["work_items"]) == (2, 340, 2, 376)
    # 21568 - 84 x 256 = 64 columns left, rounded up to what a pair stages (2 x 64): 128
    assert p["last_tile_n"] == 128
    # K > 1024: Y staged one 4 KB chunk at a time (reported as 3), two K rows per stage, and a
    # full barrier per K row (staged second operand)
    assert (p["y_blocks"], p["k_rows"], p["row_barriers"]) == (3, 2, 1)


def test_gate_glu_block_short_k():
    p = plan(1024, 21568, 256, fg.F16, gate=True)
    # K <= 512: single CTAs, 128 x 256 tiles: 8 x 85 = 680 tiles on 152 CTAs; 680 = 4 x 152 + 72
    # -> 72 tiles in 2 pieces (4 would need 288 > 152 CTAs): 608 + 144 = 752 items
    assert (p["cluster"], p["grid"], p["tiles"], p["tail_split"], p["work_items"]) == \
        (1, 152, 680, 2, 752)
    # single CTA: the last column narrowed to 64 (one 64-column box); one K row per stage
    assert (p["last_tile_n"], p["y_blocks"], p["k_rows"], p["row_barriers"]) == (64, 1, 1, 0)
    # K <= 256 on single CTAs: the bias-initialised accumulator is set by the extra MMA (2)
    assert p["bias_init"] == 2
    assert plan(1024, 21568, 256, fg.F16, gate=True, opts={"bias_mma": 1})["bias_init"] == 1
    assert plan(1024, 21568, 512, fg.F16, gate=True)["bias_init"] == 1
    assert plan(1024, 21568, 512, fg.F16, gate=True, opts={"bias_mma": 2})["bias_init"] == 2
    # an fp32 bias cannot be set by a 16-bit MMA: written by the epilogue
    assert plan(1024, 21568, 256, fg.F16 | fg.BIAS_F32, gate=True, opts={"bias_mma": 2})["bias_init"] == 1
    p = plan(1024, 21568, 1024, fg.F16, gate=True)
    # K = 1024 > 512: pairs again; 256 < K <= 1024: one 8 KB Y block per warp, one K row
    assert (p["cluster"], p["work_items"], p["y_blocks"], p["k_rows"], p["row_barriers"]) == \
        (2, 376, 1, 1, 0)
    assert p["bias_init"] == 1 and plan(1024, 21568, 4096, fg.F16, gate=True)["bias_init"] == 0


def test_fp8_operands():
    word = fg.E4M3 | fg.BIAS_F32 | fg.OUT_BF16
    p = plan(4096, 4096, 4096, word)
    # fp8 operands on pairs: the 28 tiles of the last round are cut in two like 16-bit operands'
    # (64 columns of B per CTA, in 64-byte-swizzled boxes): 228 + 56 = 284 items; two
    # 128-element K rows per stage, each on its own full barrier
    assert (p["path"], p["cluster"], p["tail_split"], p["work_items"]) == (fg.PATH_TC, 2, 2, 284)
    assert (p["k_rows"], p["row_barriers"]) == (2, 1)
    # decode-like shapes with fp8 operands take the swap-AB skinny kernel as well: 128 K elements
    # per stage, so the same K split over the cluster as 16-bit operands with half the K
    p = plan(64, 8192, 8192, word)
    q = plan(64, 8192, 4096, fg.BF16)
    assert p["path"] == fg.PATH_SKINNY and (p["grid"], p["cluster"]) == (q["grid"], q["cluster"])


@pytest.mark.parametrize("M", [1, 16, 64, 128])
def test_skinny_decode_shapes(M):
    p = plan(M, 8192, 8192, fg.BF16)
    # M <= 128 with 16-bit operands: swap-AB skinny kernel, 8192 / 128 = 64 column tiles, K split
    # until the clusters cover 2 x SMs: 2 x 152 / 64 -> 4 (at most K blocks / 4 = 32, at most 8)
    assert (p["path"], p["tiles"], p["cluster"], p["grid"], p["tail_split"]) == \
        (fg.PATH_SKINNY, 64, 4, 256, 1)


def test_small_and_ragged_shapes():
    p = plan(200, 136, 72, fg.F16 | fg.BIAS_F32)
    # K <= 512: single CTAs; tiles 2 x 1, so a grid of 2; 136 columns rounded up to 64: 192
    assert (p["path"], p["cluster"], p["grid"], p["tiles"], p["last_tile_n"]) == \
        (fg.PATH_TC, 1, 2, 2, 192)
    # a row stride that breaks TMA's 16-byte rule (K not a multiple of 8): generic path
    assert plan(200, 136, 70, fg.F16)["path"] == fg.PATH_GENERIC
    # a base pointer that is only element-aligned: generic path
    assert plan(200, 136, 72, fg.F16, a=A + 2)["path"] == fg.PATH_GENERIC
    # K = 0: the K-zero kernel; M = 0: nothing to do
    assert plan(200, 136, 0, fg.F16)["path"] == fg.PATH_KZERO
    assert plan(0, 136, 72, fg.F16)["path"] == fg.PATH_NONE


def test_options_steer_the_plan():
    # cta_pair = 1 forces single CTAs: 128 x 256 tiles, 32 x 16 = 512 on 152 CTAs;
    # 512 = 3 x 152 + 56 -> 56 tiles in 2 pieces (4 would need 224 > 152): 456 + 112 = 568 items
    p = plan(4096, 4096, 4096, fg.BF16, opts={"cta_pair": 1})
    assert (p["cluster"], p["grid"], p["tiles"], p["work_items"]) == (1, 152, 512, 568)
    # tail_split = 1 keeps whole tiles in the last round
    assert plan(4096, 4096, 4096, fg.BF16, opts={"tail_split": 1})["work_items"] == 256
    # max_ctas caps the grid: 20 CTAs = 10 pairs; 256 = 25 x 10 + 6, and 2 x 6 pieces would not
    # fit on 10 pairs, so the last round keeps whole tiles
    p = plan(4096, 4096, 4096, fg.BF16, opts={"max_ctas": 20})
    assert (p["grid"], p["tail_split"], p["work_items"]) == (20, 1, 256)
    # 24 CTAs = 12 pairs: 256 = 21 x 12 + 4 -> 4 tiles in 2 pieces: 252 + 8 = 260 items
    p = plan(4096, 4096, 4096, fg.BF16, opts={"max_ctas": 24})
    assert (p["grid"], p["tail_split"], p["work_items"]) == (24, 2, 260)
    # full_last_n runs the ragged last column at full width
    assert plan(1024, 21568, 4096, fg.F16, gate=True, opts={"full_last_n": 1})["last_tile_n"] == 256
    # the skinny split can be forced
    assert plan(16, 8192, 8192, fg.BF16, opts={"split_k": 2})["cluster"] == 2


def test_device_shape_limits_the_grid():
    # fewer resident pairs than SM pairs: the persistent grid takes what can be resident
    p = plan(4096, 4096, 4096, fg.BF16, pairs=70)
    assert (p["grid"], p["resident_pairs"]) == (140, 70)
    # a smaller device: 64 SMs = 32 pairs; 256 = 8 x 32, no partial round, no pieces
    p = plan(4096, 4096, 4096, fg.BF16, sms=64, pairs=0)
    assert (p["grid"], p["tail_split"], p["work_items"]) == (64, 1, 256)


def test_bad_device_shape_is_rejected():
    for sms, pairs in ((0, 76), (152, -1)):
        with pytest.raises(fg.FgemmError):
            plan(4096, 4096, 4096, fg.BF16, sms=sms, pairs=pairs)


@pytest.mark.parametrize("M,N,K,tiles,split", [
    (16, 2056, 4096, 17, 8),   # 17 column tiles; 2 x 152 / 17 = 17, at most 8
    (100, 520, 1024, 5, 4),    # 5 tiles; 2 x 152 / 5 = 60, at most K blocks / 4 = 16 / 4 = 4
    (16, 1032, 256, 9, 1),     # 4 K blocks: 4 / 4 = 1, no split
    (64, 136, 8, 2, 1),        # one K block: no split
])
def test_skinny_split_caps(M, N, K, tiles, split):
    p = plan(M, N, K, fg.BF16)
    assert (p["path"], p["tiles"], p["cluster"], p["grid"]) == (fg.PATH_SKINNY, tiles, split,
                                                                tiles * split)


def test_skinny_two_tiles_per_cta():
    # two 128-column tiles per CTA: 64 / 2 = 32 groups; 2 x 152 / 32 = 9, at most 8; 32 x 8 CTAs
    p = plan(16, 8192, 8192, fg.BF16, opts={"skinny_tiles": 2})
    assert (p["tail_split"], p["cluster"], p["grid"]) == (2, 8, 256)


def test_residual_and_quantised_epilogues():
    # the residual's R is staged like the gate's Y when the output is 16-bit ...
    p = plan(1024, 21568, 4096, fg.F16, epilogue=fg.EPI_RESIDUAL_RELU)
    assert (p["y_blocks"], p["k_rows"], p["row_barriers"]) == (3, 2, 1)
    # ... and read into registers (no staging, no per-row barriers) with an fp32 output
    p = plan(1024, 21568, 4096, fg.F16 | fg.OUT_F32, epilogue=fg.EPI_RESIDUAL_RELU)
    assert (p["y_blocks"], p["k_rows"], p["row_barriers"]) == (1, 2, 0)
    # fp8 output on pairs: 128-column staging rows keep pieces at 128 columns per pair, so the
    # 4096^3 tail is still cut in two (284 items); 16-bit operands: one full barrier per stage
    p = plan(4096, 4096, 4096, fg.BF16 | fg.BIAS_F32 | fg.OUT_E4M3, epilogue=fg.EPI_RELU_QUANT)
    assert (p["path"], p["tail_split"], p["work_items"], p["row_barriers"]) == (fg.PATH_TC, 2, 284, 0)


def test_unknown_option_names_are_refused():
    with pytest.raises(ValueError):
        plan(4096, 4096, 4096, fg.BF16, opts={"group": 8})  # the field is group_m
