"""The stream-K share-out of the tensor-core path's last round, on the host alone: the library's
own runs (fgemm_stream_k_run) against the rule include/fgemm.h states for them, restated here, and
the invariants the kernel relies on; then the planner's choice of stream-K (fgemm_plan_on).  No
GPU is touched."""
import os
import random
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import gemm_epilogue_gb300.binding as fg  # noqa: E402

SMS, PAIRS = 152, 76
A, B, BIAS, Y, OUT, WS = (0x10000000 + i * 0x10000000 for i in range(6))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fg.lib()


def stated_runs(u, units, sk_tiles, num_kb):
    """The rule of the header, restated: unit u takes K blocks [u S / units, (u + 1) S / units) of
    the S = sk_tiles x num_kb in (tile, K block) order, cut at tile boundaries."""
    S = sk_tiles * num_kb
    b0, b1 = u * S // units, (u + 1) * S // units
    out = []
    while b0 < b1:
        t = b0 // num_kb
        e = min(b1, (t + 1) * num_kb)
        out.append((t, b0 - t * num_kb, e - t * num_kb))
        b0 = e
    return out


def library_runs(u, units, sk_tiles, num_kb):
    out = []
    for i in range(3):
        try:
            out.append(fg.fgemm_stream_k_run(u, units, sk_tiles, num_kb, i))
        except fg.FgemmError:
            break
    return out


def check_share_out(units, sk_tiles, num_kb):
    covered = {}
    heads = {}
    parts = {}
    for u in range(units):
        mine = library_runs(u, units, sk_tiles, num_kb)
        assert [(r["tile"], r["kb0"], r["kb1"]) for r in mine] == stated_runs(u, units, sk_tiles, num_kb)
        assert 1 <= len(mine) <= 2
        for i, r in enumerate(mine):
            for kb in range(r["kb0"], r["kb1"]):
                assert (r["tile"], kb) not in covered
                covered[(r["tile"], kb)] = u
            if r["kb0"] > 0:
                # a run that does not start its tile writes slot u, and it is the unit's first
                # run: no unit waits before it has written its partial sums
                assert (r["part"], r["nsrc"], i) == (u, 0, 0)
                parts[u] = r
            else:
                assert r["part"] == -1
                if r["kb1"] < num_kb:
                    heads[r["tile"]] = (u, r)
                else:
                    assert r["nsrc"] == 0
    # every K block of every stream-K tile exactly once
    assert len(covered) == sk_tiles * num_kb
    consumed = []
    for tile, (u, h) in heads.items():
        srcs = list(range(h["src0"], h["src0"] + h["nsrc"]))
        assert srcs and srcs[0] == u + 1
        # the head's K blocks, then its sources' in the order it adds them, tile the K loop
        edge = h["kb1"]
        for s in srcs:
            p = parts[s]
            assert p["tile"] == tile and p["kb0"] == edge
            edge = p["kb1"]
        assert edge == num_kb
        consumed += srcs
    # every partial slot is read by exactly one head
    assert sorted(consumed) == sorted(parts)


@pytest.mark.parametrize("units,sk_tiles,num_kb", [
    (76, 28, 32),    # 4096^3 bf16 on 76 CTA pairs, two K rows per stage
    (76, 28, 16),    # 4096^3 fp8 operands
    (76, 44, 32),    # FFN 8192 x 14336 x 4096
    (76, 75, 16),    # one tile short of a full round
    (76, 1, 76),     # one tile: every unit one K block
    (152, 56, 16),   # single CTAs
    (5, 3, 2),       # tiny: runs of one or two K blocks
])
def test_share_out_of_measured_and_edge_shapes(units, sk_tiles, num_kb):
    check_share_out(units, sk_tiles, num_kb)


def test_share_out_random_shapes():
    rnd = random.Random(7)
    for _ in range(150):
        units = rnd.randint(2, 160)
        sk_tiles = rnd.randint(1, units - 1)
        num_kb = rnd.randint(max(1, -(-units // sk_tiles)), 80)
        check_share_out(units, sk_tiles, num_kb)


def test_share_out_rejects_what_it_cannot_deal():
    for args in ((0, 76, 28, 32, 2),    # no run 2
                 (76, 76, 28, 32, 0),   # u out of range
                 (0, 76, 76, 32, 0),    # sk_tiles must be below units
                 (0, 76, 2, 30, 0),     # fewer K blocks than units
                 (0, 0, 1, 1, 0)):
        with pytest.raises(fg.FgemmError):
            fg.fgemm_stream_k_run(*args)


def plan(M, N, K, dtype, opts=None, gate=False, epilogue=None):
    return fg.fgemm_plan_on(A, B, BIAS, Y if gate else None, OUT, M, N, K, dtype, SMS, PAIRS,
                            gate=gate, opts=opts, epilogue=epilogue)


def sk_items(full, units, sk_tiles, num_kb):
    return full + sum(len(stated_runs(u, units, sk_tiles, num_kb)) for u in range(units))


# 256 x 256 tiles on 76 pairs: 16 x 16 = 256 tiles = 3 x 76 + 28; a 16-bit stage is two K rows of
# 64 elements, so K = 4096 is 32 K blocks per tile.  Workspace: the flag area and 152 CTA slots of
# 128 x 256 fp32.
SQ_WS = fg.SK_FLAG_BYTES + 152 * 128 * 256 * 4


def test_square_takes_stream_k_with_a_workspace():
    p = plan(4096, 4096, 4096, fg.BF16, opts={"workspace": WS, "workspace_bytes": SQ_WS})
    assert (p["sk_tiles"], p["tail_split"], p["sk_workspace_bytes"]) == (28, 1, SQ_WS)
    assert p["work_items"] == sk_items(228, 76, 28, 32)


def test_square_without_a_workspace_keeps_the_column_pieces():
    p = plan(4096, 4096, 4096, fg.BF16)
    # the workspace it would need is reported all the same
    assert (p["sk_tiles"], p["tail_split"], p["work_items"], p["sk_workspace_bytes"]) == \
        (0, 2, 284, SQ_WS)
    # one byte short: no stream-K in automatic mode, an error when it is asked for
    small = {"workspace": WS, "workspace_bytes": SQ_WS - 1}
    assert plan(4096, 4096, 4096, fg.BF16, opts=small)["sk_tiles"] == 0
    with pytest.raises(fg.FgemmError) as e:
        plan(4096, 4096, 4096, fg.BF16, opts=dict(small, stream_k=1))
    assert e.value.status == fg.ERR_WORKSPACE


def test_stream_k_switches():
    ws = {"workspace": WS, "workspace_bytes": SQ_WS}
    assert plan(4096, 4096, 4096, fg.BF16, opts=dict(ws, stream_k=2))["sk_tiles"] == 0
    assert plan(4096, 4096, 4096, fg.BF16, opts=dict(ws, stream_k=1))["sk_tiles"] == 28
    # a bias-initialised accumulator asked for: automatic mode leaves stream-K off, forcing both
    # is refused (partial sums must not hold the bias)
    assert plan(4096, 4096, 4096, fg.BF16, opts=dict(ws, bias_init=1))["sk_tiles"] == 0
    with pytest.raises(fg.FgemmError) as e:
        plan(4096, 4096, 4096, fg.BF16, opts=dict(ws, bias_init=1, stream_k=1))
    assert e.value.status == fg.ERR_INVALID_VALUE
    # the workspace must be 256-byte aligned
    with pytest.raises(fg.FgemmError) as e:
        plan(4096, 4096, 4096, fg.BF16, opts={"workspace": WS + 16, "workspace_bytes": SQ_WS})
    assert e.value.status == fg.ERR_MISALIGNED


def test_shapes_that_do_not_qualify():
    ws = {"workspace": WS, "workspace_bytes": 1 << 30}
    with pytest.raises(fg.FgemmError):
        plan(4096, 4096, 1024, fg.BF16, opts=dict(ws, stream_k=1))
    # K = 1024 on pairs: 8 K blocks per tile, below 16
    assert plan(4096, 4096, 1024, fg.BF16, opts=ws)["sk_tiles"] == 0
    # a grid that divides the tiles has no partial round: 256 tiles on 64 pairs
    assert plan(4096, 4096, 4096, fg.BF16, opts=dict(ws, max_ctas=128))["sk_tiles"] == 0


def test_other_shapes_that_qualify():
    ws = {"workspace": WS, "workspace_bytes": 1 << 30}
    # fp8 operands: two 128-element K rows per stage, K = 4096 is 16 K blocks
    p = plan(4096, 4096, 4096, fg.E4M3 | fg.BIAS_F32 | fg.OUT_BF16, opts=ws)
    assert (p["sk_tiles"], p["work_items"]) == (28, sk_items(228, 76, 28, 16))
    # FFN 8192 x 14336 x 4096: 32 x 56 = 1792 tiles = 23 x 76 + 44
    p = plan(8192, 14336, 4096, fg.BF16, opts=ws)
    assert (p["sk_tiles"], p["work_items"]) == (44, sk_items(1748, 76, 44, 32))
    # the GLU block's gate: 4 x 85 = 340 tiles = 4 x 76 + 36, K = 4096 in 32 K blocks (two K rows
    # per stage with Y staged one chunk at a time); with an fp32 output Y goes to registers
    for w in (fg.F16, fg.F16 | fg.OUT_F32):
        p = plan(1024, 21568, 4096, w, gate=True, opts=ws)
        assert (p["sk_tiles"], p["work_items"]) == (36, sk_items(304, 76, 36, 32))
