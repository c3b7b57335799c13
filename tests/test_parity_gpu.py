"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs."""

import numpy as np
import pytest

import oracle
from conftest import parse_matrix, read_golden
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import (BF16, E4M3, F16, F32, check_close, check_guarded, down, dtype_word,
                      guarded_out, sample_rows, torch_dtype, up)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gemm_epilogue_gb300.binding as fg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemm_epilogue_gb300 import build
    build.build()
    oracle.build()
    fg.lib()
    yield
    assert fg.fgemm_device_status() == 0


def run_fused(p, M, N, K, ab, bt, ot, gate=False, opts=None, out=None):
    A, B = up(p.A, ab), up(p.B, ab)
    bias = up(p.bias, bt)
    Y = up(p.Y, ab) if gate else None
    if out is None:
        out = torch.empty(M, N, dtype={F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}[ot],
                          device="cuda")
    w = dtype_word(ab, bt, ot)
    if gate:
        path = fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, w, opts=opts)
    else:
        path = fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, w, opts=opts)
    torch.cuda.synchronize()
    return out, path


def oracle_run(p, M, N, K, ab, bt, ot, gate=False, rows=None, y_type=None):
    if gate:
        return oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, ab, bt, ot, rows=rows,
                                 y_type=y_type)
    return oracle.bias_relu(p.A, p.B, p.bias, M, N, K, ab, bt, ot, rows=rows)


# ------------------------------------------------------------ exact small cases --

@pytest.mark.parametrize("ab,bt,ot", [(F16, F16, F16), (BF16, BF16, BF16), (F16, F32, F32)])
def test_worked_example(ab, bt, ot):
    g = read_golden("worked_example_2x2.txt")
    A = oracle.encode(np.array(parse_matrix(g["A"])), ab)
    B = oracle.encode(np.array(parse_matrix(g["B"])), ab)
    bias = oracle.encode(np.array(parse_matrix(g["bias"])[0]), bt)
    p = gen.Inputs(A, B, bias, None)
    out, path = run_fused(p, 2, 2, 2, ab, bt, ot)
    assert path == fg.PATH_GENERIC
    assert np.array_equal(oracle.decode(down(out, ot), ot), np.array(parse_matrix(g["relu"])))


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("ab,bt,ot", [(F16, F32, F16), (BF16, BF16, BF16), (BF16, BF16, F32)])
def test_k_zero(gate, ab, bt, ot):
    M, N = 37, 70
    p = gen.random_problem(M, N, 0, ab, bt, seed=1, gate=gate)
    out, path = run_fused(gen.Inputs(None, None, p.bias, p.Y), M, N, 0, ab, bt, ot, gate=gate)
    assert path == fg.PATH_KZERO
    ref = oracle_run(gen.Inputs(None, None, p.bias, p.Y), M, N, 0, ab, bt, ot, gate=gate)
    assert np.array_equal(down(out, ot), ref.out)


@pytest.mark.parametrize("K", [1, 3])
def test_k1_k3_fused_matches_oracle_and_unfused_chain(K):
    # "Epilogue concept", "Things that break": same shape at K = 1 and K = 3.
    M, N = 37, 45
    p = gen.integer_problem(M, N, K, F16, F16, seed=K)
    out, _ = run_fused(p, M, N, K, F16, F16, F16)
    ref = oracle_run(p, M, N, K, F16, F16, F16)
    assert np.array_equal(down(out, F16), ref.out)
    ws_bytes = fg.fgemm_unfused_workspace_bytes(M, N, fg.F16, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out2 = torch.empty(M, N, dtype=torch.float16, device="cuda")
    fg.fgemm_unfused_bias_relu(up(p.A, F16), up(p.B, F16), up(p.bias, F16), out2, M, N, K, fg.F16,
                               ws, ws_bytes, 1)
    torch.cuda.synchronize()
    assert np.array_equal(down(out2, F16), ref.out)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 2), (7, 9, 40), (17, 33, 13), (40, 40, 39),
                                   (65, 3, 31), (2, 129, 17)])
def test_brute_force_ragged_generic_bit_exact(M, N, K):
    for ab, bt, ot in ((F16, F16, F16), (BF16, F32, BF16)):
        p = gen.integer_problem(M, N, K, ab, bt, seed=M + N + K)
        out, path = run_fused(p, M, N, K, ab, bt, ot)
        assert path == fg.PATH_GENERIC
        assert np.array_equal(down(out, ot), oracle_run(p, M, N, K, ab, bt, ot).out)
        g = gen.integer_problem(M, N, K, ab, bt, seed=M * N + K, gate=True)
        out, _ = run_fused(g, M, N, K, ab, bt, ot, gate=True)
        assert np.array_equal(down(out, ot), oracle_run(g, M, N, K, ab, bt, ot, gate=True).out)


# ------------------------------------------------------ tensor-core path, exact --

TC_SHAPES = [(1, 8, 8), (128, 256, 64), (200, 136, 72), (129, 264, 136), (300, 520, 200),
             (77, 1032, 24), (513, 264, 256)]


@pytest.mark.parametrize("M,N,K", TC_SHAPES)
@pytest.mark.parametrize("ab", [F16, BF16])
@pytest.mark.parametrize("pair", [1, 2])
def test_tc_integer_bit_exact(M, N, K, ab, pair):
    # Small integers: every partial sum is exact in fp32, so the only rounding is the final one
    # and the tensor-core result must equal the oracle bit for bit.  Shapes are ragged against the
    # 128 x 256 x 64 tile (single CTA) and the 256 x 256 tile (CTA pair) in M, N and K.
    p = gen.integer_problem(M, N, K, ab, ab, seed=M * 7 + N + K)
    out, path = run_fused(p, M, N, K, ab, ab, ab, opts={"path": fg.PATH_TC, "cta_pair": pair})
    assert path == fg.PATH_TC
    ref = oracle_run(p, M, N, K, ab, ab, ab)
    got = down(out, ab)
    if not np.array_equal(got, ref.out):
        bad = np.argwhere(got != ref.out)
        pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")


@pytest.mark.parametrize("M,N,K", [(200, 136, 72), (300, 520, 200), (777, 1288, 328)])
@pytest.mark.parametrize("pair", [1, 2])
def test_tc_gate_integer_bit_exact(M, N, K, pair):
    for ab, ot in ((F16, F16), (BF16, F32)):
        p = gen.integer_problem(M, N, K, ab, ab, seed=K, gate=True)
        out, path = run_fused(p, M, N, K, ab, ab, ot, gate=True, opts={"cta_pair": pair})
        assert path == fg.PATH_TC
        assert np.array_equal(down(out, ot), oracle_run(p, M, N, K, ab, ab, ot, gate=True).out)


@pytest.mark.parametrize("bt,ot", [(F32, F32), (F32, F16), (F16, F32)])
def test_tc_bias_and_output_types(bt, ot):
    M, N, K = 150, 392, 96
    p = gen.integer_problem(M, N, K, F16, bt, seed=5)
    out, path = run_fused(p, M, N, K, F16, bt, ot)
    assert path == fg.PATH_TC
    assert np.array_equal(down(out, ot), oracle_run(p, M, N, K, F16, bt, ot).out)


# ------------------------------------------------------------ skinny-M path --

SKINNY_SHAPES = [(1, 8, 8, 1), (1, 136, 72, 2), (5, 264, 520, 3), (16, 1032, 2048, 4),
                 (33, 392, 256, 2), (64, 136, 8, 4), (100, 520, 1024, 8), (128, 1032, 512, 2)]


@pytest.mark.parametrize("M,N,K,split", SKINNY_SHAPES)
@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("tiles", [1, 2])
def test_skinny_integer_bit_exact(M, N, K, split, gate, tiles):
    # split K over a cluster; (64, 136, 8, 4) leaves some CTAs of the cluster with no K block;
    # tiles = 2 gives each CTA two 128-column tiles sharing A (N = 136 leaves the second ragged)
    for ab, bt, ot in ((BF16, BF16, BF16), (F16, F32, F32)):
        p = gen.integer_problem(M, N, K, ab, bt, seed=M + N + K + split, gate=gate)
        out, path = run_fused(p, M, N, K, ab, bt, ot, gate=gate,
                              opts={"split_k": split, "skinny_tiles": tiles})
        assert path == fg.PATH_SKINNY
        ref = oracle_run(p, M, N, K, ab, bt, ot, gate=gate)
        got = down(out, ot)
        if not np.array_equal(got, ref.out):
            bad = np.argwhere(got != ref.out)
            pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")


@pytest.mark.parametrize("M,N,K,tiles", [(64, 520, 4096, 1), (128, 264, 2048, 1), (16, 1032, 8192, 2)])
def test_skinny_single_cta_long_k_bit_exact(M, N, K, tiles):
    # split 1 (no cluster) with long main loops: the epilogue warps synchronise among themselves
    # while the producer and MMA lanes may still be in their loops
    p = gen.integer_problem(M, N, K, BF16, BF16, seed=M + N + K)
    out, path = run_fused(p, M, N, K, BF16, BF16, BF16, opts={"split_k": 1, "skinny_tiles": tiles})
    assert path == fg.PATH_SKINNY
    ref = oracle_run(p, M, N, K, BF16, BF16, BF16)
    got = down(out, BF16)
    if not np.array_equal(got, ref.out):
        bad = np.argwhere(got != ref.out)
        pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")


@pytest.mark.parametrize("M,N,K,opts,want_path", [
    (300, 520, 200, None, 1),            # tensor cores, single CTAs, ragged last column
    (700, 1800, 1104, None, 1),          # CTA pairs, last column narrowed to 128 of 256
    (16, 1032, 512, None, 2),            # skinny, ragged last 128-column tile
    (7, 9, 13, None, 3),                 # generic
])
@pytest.mark.parametrize("gate", [False, True])
def test_bias_padded_with_nan_past_n(M, N, K, opts, want_path, gate):
    # "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "Pitfalls": the bias load must be
    # masked with j < N.  The bias buffer runs on past N with NaNs; a read past the end that leaked
    # into a stored column would show up as a NaN in out.
    p = gen.integer_problem(M, N, K, BF16, BF16, seed=M + N + K, gate=gate)
    A, B = up(p.A, BF16), up(p.B, BF16)
    padded = torch.full((N + 512,), float("nan"), dtype=torch.bfloat16, device="cuda")
    padded[:N] = up(p.bias, BF16)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w = dtype_word(BF16, BF16, BF16)
    if gate:
        path = fg.fgemm_addmm_gate_ex(A, B, padded, up(p.Y, BF16), out, M, N, K, w, opts=opts)
    else:
        path = fg.fgemm_bias_relu_ex(A, B, padded, out, M, N, K, w, opts=opts)
    torch.cuda.synchronize()
    assert path == want_path
    assert not torch.isnan(out).any()
    # by value: with the bias-initialised accumulator an exact zero may come out as -0
    assert _same_values(down(out, BF16), oracle_run(p, M, N, K, BF16, BF16, BF16, gate=gate).out,
                        BF16)


def test_skinny_auto_split_and_coverage():
    M, N, K = 16, 2056, 4096
    p = gen.random_problem(M, N, K, BF16, BF16, seed=12)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + M * N].view(M, N)
    _, path = run_fused(p, M, N, K, BF16, BF16, BF16, out=out)
    assert path == fg.PATH_SKINNY
    b = buf.cpu()
    assert torch.isnan(b[:guard]).all() and torch.isnan(b[guard + M * N:]).all()
    ref = oracle_run(p, M, N, K, BF16, BF16, BF16)
    check_close(down(out, BF16), ref, K, BF16, bias64=oracle.decode(p.bias, BF16), what="skinny")


def test_skinny_matches_square_tile_path():
    M, N, K = 128, 1024, 1024
    p = gen.random_problem(M, N, K, F16, F16, seed=13)
    a, _ = run_fused(p, M, N, K, F16, F16, F16, opts={"path": fg.PATH_SKINNY})
    b, _ = run_fused(p, M, N, K, F16, F16, F16, opts={"path": fg.PATH_TC})
    ref = oracle_run(p, M, N, K, F16, F16, F16)
    for x in (a, b):
        check_close(down(x, F16), ref, K, F16, bias64=oracle.decode(p.bias, F16), what="skinny/tc")


# ------------------------------------------------------------- residual add --

RESID_CASES = [  # M, N, K, opts, expected path
    (300, 520, 200, {"cta_pair": 2}, 1), (300, 520, 200, {"cta_pair": 1}, 1),
    (300, 520, 2048, {"cta_pair": 2}, 1),  # long K on pairs: R staged a chunk at a time, row barriers
    (777, 1288, 328, None, 1), (16, 1032, 512, None, 2), (100, 264, 72, {"split_k": 3}, 2),
    (7, 9, 13, None, 3), (37, 70, 0, None, 4)]


@pytest.mark.parametrize("M,N,K,opts,want_path", RESID_CASES)
def test_residual_integer_bit_exact(M, N, K, opts, want_path):
    # "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "Variants": residual tile added after
    # the K loop, before the activation; every path, 16-bit and fp32 outputs
    for ab, ot in ((BF16, BF16), (F16, F32)):
        p = gen.integer_problem(M, N, K, ab, ab, seed=M + N + K, gate=True)  # Y serves as R
        A = up(p.A, ab) if K else None
        B = up(p.B, ab) if K else None
        bias, R = up(p.bias, ab), up(p.Y, ab)
        out = torch.empty(M, N, dtype={F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}[ot],
                          device="cuda")
        path = fg.fgemm_bias_residual_relu_ex(A, B, bias, R, out, M, N, K, dtype_word(ab, ab, ot),
                                              opts=opts)
        torch.cuda.synchronize()
        assert path == want_path
        ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ot)
        assert np.array_equal(down(out, ot), ref.out)


def test_residual_random_tolerance_and_guards():
    M, N, K = 513, 776, 1024
    p = gen.random_problem(M, N, K, BF16, BF16, seed=15, gate=True)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + M * N].view(M, N)
    fg.fgemm_bias_residual_relu(up(p.A, BF16), up(p.B, BF16), up(p.bias, BF16), up(p.Y, BF16), out,
                                M, N, K, fg.BF16)
    torch.cuda.synchronize()
    b = buf.cpu()
    assert torch.isnan(b[:guard]).all() and torch.isnan(b[guard + M * N:]).all()
    ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, BF16, BF16, BF16)
    check_close(down(out, BF16), ref, K, BF16, bias64=oracle.decode(p.bias, BF16) + 0.0,
                Y64=None, what="residual")


# ------------------------------------------------------- quantized fp8 output --

QUANT_CASES = [  # M, N, K, opts, expected path
    (300, 528, 200, {"cta_pair": 2}, 1), (300, 528, 200, {"cta_pair": 1, "max_ctas": 20}, 1),
    (777, 1296, 328, None, 1), (16, 1040, 512, None, 2), (100, 272, 72, {"split_k": 3}, 2),
    (7, 37, 13, None, 3), (300, 520, 200, None, 3), (37, 80, 0, None, 4)]


def _run_quant(p, M, N, K, ab, bt, scale, opts=None):
    A = up(p.A, ab) if K else None
    B = up(p.B, ab) if K else None
    out = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    w = (fg.F16 if ab == F16 else fg.BF16) | (fg.BIAS_F32 if bt == F32 else 0) | fg.OUT_E4M3
    path = fg.fgemm_bias_relu_quant_ex(A, B, up(p.bias, bt), out, M, N, K, w, scale, opts=opts)
    torch.cuda.synchronize()
    return out.cpu().numpy(), path


@pytest.mark.parametrize("M,N,K,opts,want_path", QUANT_CASES)
def test_quant_integer_bit_exact(M, N, K, opts, want_path):
    # "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", "Variants": matmul + quantized output.
    # Integer inputs and power-of-two scales keep every value exact until the fp8 rounding, which
    # both sides then take from the same number (saturating at 448 for the large sums).
    for ab, bt, scale in ((BF16, BF16, 0.25), (F16, F32, 2.0)):
        p = gen.integer_problem(M, N, K, ab, bt, seed=M + N + K)
        got, path = _run_quant(p, M, N, K, ab, bt, scale, opts)
        assert path == want_path
        ref = oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, ab, bt, scale)
        if not np.array_equal(got, ref.out):
            bad = np.argwhere(got != ref.out)
            pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")


def test_quant_random_within_one_fp8_step():
    M, N, K = 513, 784, 1024
    p = gen.random_problem(M, N, K, BF16, BF16, seed=16, scale=K ** -0.25)
    scale = 3.7
    got, path = _run_quant(p, M, N, K, BF16, BF16, scale)
    assert path == fg.PATH_TC
    ref = oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, BF16, BF16, scale)
    g = oracle.decode(got, E4M3)
    r = oracle.decode(ref.out, E4M3)
    exact = ref.ref
    # fp8 spacing at |exact| (3 fraction bits, subnormal spacing 2^-9)
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -6))) - 3)
    assert np.all(np.abs(g - r) <= step + 1e-12)
    assert np.mean(g == r) > 0.99


# ------------------------------------------------------------ fp8 operands --

FP8_CASES = [  # M, N, K, opts, expected path
    (300, 528, 256, {"cta_pair": 2}, 1), (300, 528, 256, {"cta_pair": 1, "max_ctas": 20}, 1),
    (777, 1296, 336, None, 1), (96, 1040, 512, None, 2), (7, 40, 24, None, 3),
    (300, 520, 200, None, 3)]


@pytest.mark.parametrize("M,N,K,opts,want_path", FP8_CASES)
def test_fp8_operands_integer_bit_exact(M, N, K, opts, want_path):
    # fp8 e4m3 A and B (tcgen05 kind::f8f6f4 on the tensor-core path): integer inputs are exact in
    # e4m3 and every sum is exact in fp32, so the only rounding is the output's.
    for bt, ot in ((F32, BF16), (BF16, F32)):
        p = gen.integer_problem(M, N, K, E4M3, bt, seed=M + K)
        out = torch.empty(M, N, dtype={BF16: torch.bfloat16, F32: torch.float32}[ot], device="cuda")
        path = fg.fgemm_bias_relu_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, bt), out, M, N, K,
                                     dtype_word(E4M3, bt, ot), opts=opts)
        torch.cuda.synchronize()
        assert path == want_path
        ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, bt, ot)
        got = down(out, ot)
        if not np.array_equal(got, ref.out):
            bad = np.argwhere(got != ref.out)
            pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")


# fp8 operands on CTA pairs with the last round cut into 128-column pieces: 64 columns of B per
# CTA, staged as 64-byte-swizzled boxes (M, N, K, grid cap, epilogue)
FP8_PIECE_CASES = [(1280, 1024, 2048, 16, "relu"), (1000, 848, 1152, 10, "relu"),
                   (1280, 1024, 1024, 16, "gate"), (777, 1296, 1344, 14, "quant")]


@pytest.mark.parametrize("M,N,K,mc,epi", FP8_PIECE_CASES)
def test_fp8_pair_column_pieces_integer_bit_exact(M, N, K, mc, epi):
    opts = {"cta_pair": 2, "max_ctas": mc}
    gate = epi == "gate"
    p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + N, gate=gate, y_type=F16 if gate else None)
    A, B, bias = up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32)
    if epi == "quant":
        ot, word = E4M3, fg.E4M3 | fg.BIAS_F32 | fg.OUT_E4M3
    else:
        ot = F16 if gate else BF16
        word = dtype_word(E4M3, F32, ot, F16 if gate else None)
    Y = up(p.Y, F16) if gate else None
    probe = torch.empty(M, N, dtype=torch.uint8 if ot == E4M3 else torch_dtype(ot), device="cuda")
    plan = fg.fgemm_plan(A, B, bias, Y, probe, M, N, K, word, gate=gate, opts=opts,
                         epilogue=fg.EPI_RELU_QUANT if epi == "quant" else None)
    assert plan["cluster"] == 2 and plan["tail_split"] == 2, plan
    out, buf = guarded_out(M, N, ot)
    if gate:
        fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, word, opts=opts)
        ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, E4M3, F32, ot, y_type=F16)
    elif epi == "quant":
        fg.fgemm_bias_relu_quant_ex(A, B, bias, out, M, N, K, word, 0.5, opts=opts)
        ref = oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, E4M3, F32, 0.5)
    else:
        fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, word, opts=opts)
        ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, F32, ot)
    torch.cuda.synchronize()
    check_guarded(buf, M, N, ot, epi)
    got = down(out, ot)
    if not _same_values(got, ref.out, ot):
        bad = np.argwhere(got != ref.out)
        pytest.fail(f"{epi}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


def test_fp8_operands_quantized_output_bit_exact():
    M, N, K = 300, 528, 256
    p = gen.integer_problem(M, N, K, E4M3, F32, seed=9)
    out = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    fg.fgemm_bias_relu_quant(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), out, M, N, K,
                             fg.E4M3 | fg.BIAS_F32 | fg.OUT_E4M3, 0.5)
    torch.cuda.synchronize()
    ref = oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, E4M3, F32, 0.5)
    assert np.array_equal(out.cpu().numpy(), ref.out)


def test_fp8_operands_random_tolerance():
    M, N, K = 1000, 2064, 2048
    p = gen.random_problem(M, N, K, E4M3, F32, seed=17, scale=K ** -0.25)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    path = fg.fgemm_bias_relu_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), out, M, N, K,
                                 dtype_word(E4M3, F32, BF16))
    torch.cuda.synchronize()
    assert path == fg.PATH_TC
    ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, F32, BF16)
    check_close(down(out, BF16), ref, K, BF16, bias64=oracle.decode(p.bias, F32), what="fp8")


FP8_GATE_CASES = [  # M, N, K, opts, expected path
    (300, 528, 256, {"cta_pair": 2}, 1), (300, 528, 256, {"cta_pair": 1, "max_ctas": 20}, 1),
    (777, 1296, 1344, None, 1),  # K > 1024: CTA pairs, Y staged one 4 KB chunk at a time
    (513, 1040, 640, None, 1),   # 512 < K <= 1024: CTA pairs, one Y block per warp
    (96, 1040, 512, None, 2),    # M <= 128: the swap-AB skinny kernel
    (7, 40, 24, None, 3), (300, 520, 200, None, 3)]  # N not a multiple of 16: CUDA cores


@pytest.mark.parametrize("M,N,K,opts,want_path", FP8_GATE_CASES)
def test_fp8_gate_and_residual_integer_bit_exact(M, N, K, opts, want_path):
    # "Optimizing GEMM + Activation on CDNA4 with TLX", "Future Work" (FP8 precision): the
    # projection on fp8 e4m3 operands, Y (or R) and the output 16-bit.  Integer inputs are exact
    # in e4m3 and every sum is exact in fp32, so the only rounding is the output's.
    for yt, ot in ((F16, F16), (BF16, BF16), (F16, F32)):
        for epi in ("gate", "residual"):
            p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + K + yt, gate=True, y_type=yt)
            A, B, bias, Y = up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), up(p.Y, yt)
            out = torch.full((M, N), float("nan"), dtype=torch_dtype(ot), device="cuda")
            word = dtype_word(E4M3, F32, ot, yt)
            if epi == "gate":
                path = fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, word, opts=opts)
                ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, E4M3, F32, ot, y_type=yt)
            else:
                path = fg.fgemm_bias_residual_relu_ex(A, B, bias, Y, out, M, N, K, word, opts=opts)
                ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, E4M3, F32, ot,
                                                y_type=yt)
            torch.cuda.synchronize()
            assert path == want_path, (epi, yt, ot)
            got = down(out, ot)
            if not _same_values(got, ref.out, ot):
                bad = np.argwhere(oracle.decode(got, ot) != oracle.decode(ref.out, ot))
                pytest.fail(f"{epi} Y {yt} out {ot}: {len(bad)} mismatches, first at {bad[:5].tolist()}")


def test_fp8_gate_k_zero_and_16_bit_operands_with_another_y_type():
    # K = 0: out = bias + bias * Y with Y of its own type; and 16-bit operands with a Y type of
    # the other 16-bit format (the output then takes Y's type)
    M, N = 37, 80
    p = gen.integer_problem(M, N, 0, E4M3, F32, seed=3, gate=True, y_type=BF16)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    path = fg.fgemm_addmm_gate_ex(None, None, up(p.bias, F32), up(p.Y, BF16), out, M, N, 0,
                                  dtype_word(E4M3, F32, BF16, BF16))
    torch.cuda.synchronize()
    assert path == fg.PATH_KZERO
    ref = oracle.addmm_gate(None, None, p.bias, p.Y, M, N, 0, E4M3, F32, BF16, y_type=BF16)
    assert _same_values(down(out, BF16), ref.out, BF16)
    for (M, N, K), want_path in (((300, 520, 200), 1), ((16, 1032, 512), 2), ((7, 44, 9), 3)):
        p = gen.integer_problem(M, N, K, F16, F16, seed=K, gate=True, y_type=BF16)
        out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        path = fg.fgemm_addmm_gate_ex(up(p.A, F16), up(p.B, F16), up(p.bias, F16), up(p.Y, BF16),
                                      out, M, N, K, dtype_word(F16, F16, BF16, BF16))
        torch.cuda.synchronize()
        assert path == want_path
        ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, BF16, y_type=BF16)
        assert _same_values(down(out, BF16), ref.out, BF16), (M, N, K)


def test_fp8_operands_refused_where_unsupported():
    # the gate with fp8 operands needs the Y type: without it Y would be fp8, which is refused
    st = fg.call_status("fgemm_addmm_gate", None, None, None, None, None, 4, 4, 4,
                        fg.E4M3 | fg.BIAS_F32 | fg.OUT_BF16, None)
    assert st == fg.ERR_UNSUPPORTED_DTYPE
    st = fg.call_status("fgemm_bias_relu", None, None, None, None, 4, 4, 4, fg.E4M3, None)
    assert st == fg.ERR_UNSUPPORTED_DTYPE


# ------------------------------------- narrowed last tile, bias-initialised accumulator --

@pytest.mark.parametrize("N", [264, 320, 328, 384, 392, 448, 456, 504, 512])
@pytest.mark.parametrize("pair", [1, 2])
def test_narrowed_last_tile_integer_bit_exact(N, pair):
    # "Optimizing GEMM + Activation on CDNA4 with TLX", "Future Work": a last N tile narrower than
    # 256 columns.  Every remainder class of N mod 256 against the narrowing granule (64 columns on
    # one CTA, 128 on a pair), with the gate; the full-width diagnostic must give the same bits.
    M, K = 300, 136
    gran = 64 * pair
    left = N - (N - 1) // 256 * 256
    want_width = min(256, -(-left // gran) * gran)
    for gate in (False, True):
        p = gen.integer_problem(M, N, K, F16, F16, seed=N + pair, gate=gate)
        opts = {"path": fg.PATH_TC, "cta_pair": pair}
        plan = fg.fgemm_plan(up(p.A, F16), up(p.B, F16), up(p.bias, F16),
                             up(p.Y, F16) if gate else None,
                             torch.empty(M, N, dtype=torch.float16, device="cuda"), M, N, K, fg.F16,
                             gate=gate, opts=opts)
        assert plan["last_tile_n"] == want_width
        out, path = run_fused(p, M, N, K, F16, F16, F16, gate=gate, opts=opts)
        assert path == fg.PATH_TC
        ref = oracle_run(p, M, N, K, F16, F16, F16, gate=gate)
        assert np.array_equal(down(out, F16), ref.out)
        full, _ = run_fused(p, M, N, K, F16, F16, F16, gate=gate, opts=dict(opts, full_last_n=1))
        assert torch.equal(full, out)


BIAS_INIT_CASES = [  # M, N, K, opts
    (300, 520, 200, {"cta_pair": 2}), (300, 520, 200, {"cta_pair": 1}),
    (700, 1800, 200, {"cta_pair": 1, "max_ctas": 44}), (700, 1800, 200, {"cta_pair": 2, "max_ctas": 20}),
    (129, 264, 8, None), (1, 8, 64, None)]


Y_BLOCK_CASES = [  # M, N, K, max_ctas (0 = every SM)
    (300, 520, 200, 0), (700, 1800, 200, 20), (1000, 2056, 1096, 0), (513, 1288, 64, 12)]


@pytest.mark.parametrize("M,N,K,max_ctas", Y_BLOCK_CASES)
@pytest.mark.parametrize("y_blocks", [1, 2, 3])
def test_staged_y_blocks_integer_bit_exact(M, N, K, max_ctas, y_blocks):
    # The gate's Y (and the residual's R) staged one or two tiles ahead per epilogue warp, or one
    # 32 x 64 chunk at a time (3), on CTA pairs; tail pieces and the narrowed last tile included.
    opts = {"path": fg.PATH_TC, "cta_pair": 2, "max_ctas": max_ctas, "y_blocks": y_blocks}
    p = gen.integer_problem(M, N, K, F16, F16, seed=M + K + y_blocks, gate=True)
    plan = fg.fgemm_plan(up(p.A, F16), up(p.B, F16), up(p.bias, F16), up(p.Y, F16),
                         torch.empty(M, N, dtype=torch.float16, device="cuda"), M, N, K, fg.F16,
                         gate=True, opts=opts)
    assert plan["y_blocks"] == y_blocks
    auto = fg.fgemm_plan(up(p.A, F16), up(p.B, F16), up(p.bias, F16), up(p.Y, F16),
                         torch.empty(M, N, dtype=torch.float16, device="cuda"), M, N, K, fg.F16,
                         gate=True, opts={"cta_pair": 2})
    assert auto["y_blocks"] == (3 if K > 1024 else 2 if K <= 256 else 1)
    assert auto["k_rows"] == (2 if K > 1024 else 1)
    out, path = run_fused(p, M, N, K, F16, F16, F16, gate=True, opts=opts)
    assert path == fg.PATH_TC
    assert np.array_equal(down(out, F16), oracle_run(p, M, N, K, F16, F16, F16, gate=True).out)
    res = torch.empty(M, N, dtype=torch.float16, device="cuda")
    fg.fgemm_bias_residual_relu_ex(up(p.A, F16), up(p.B, F16), up(p.bias, F16), up(p.Y, F16), res,
                                   M, N, K, fg.F16, opts=opts)
    torch.cuda.synchronize()
    ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, F16)
    assert np.array_equal(down(res, F16), ref.out)


K_ROW_CASES = [  # M, N, K, max_ctas (0 = every SM)
    (300, 520, 200, 0), (700, 1800, 72, 20), (513, 1288, 136, 12), (257, 264, 1096, 0)]


@pytest.mark.parametrize("M,N,K,max_ctas", K_ROW_CASES)
@pytest.mark.parametrize("k_rows", [1, 2])
def test_k_rows_per_stage_integer_bit_exact(M, N, K, max_ctas, k_rows):
    # One or two 128-byte K rows per ring stage on CTA pairs, with K not a multiple of a stage
    # (the last stage's second row lies past K), tail pieces and the narrowed last tile.
    opts = {"path": fg.PATH_TC, "cta_pair": 2, "max_ctas": max_ctas, "k_rows": k_rows}
    p = gen.integer_problem(M, N, K, BF16, BF16, seed=M + K + k_rows)
    plan = fg.fgemm_plan(up(p.A, BF16), up(p.B, BF16), up(p.bias, BF16), None,
                         torch.empty(M, N, dtype=torch.bfloat16, device="cuda"), M, N, K, fg.BF16,
                         opts=opts)
    assert plan["k_rows"] == k_rows
    out, path = run_fused(p, M, N, K, BF16, BF16, BF16, opts=opts)
    assert path == fg.PATH_TC
    assert np.array_equal(down(out, BF16), oracle_run(p, M, N, K, BF16, BF16, BF16).out)
    p = gen.integer_problem(M, N, K, F16, F32, seed=M + 1)
    out, _ = run_fused(p, M, N, K, F16, F32, F32, opts=opts)
    assert np.array_equal(down(out, F32), oracle_run(p, M, N, K, F16, F32, F32).out)
    if N % 16 == 0:
        p = gen.integer_problem(M, N, K, BF16, F32, seed=M + 2)
        got, _ = _run_quant(p, M, N, K, BF16, F32, 0.25, opts)
        assert np.array_equal(got, oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, BF16, F32, 0.25).out)
    if N % 16 == 0 and K % 16 == 0:
        p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + 3)
        out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        fg.fgemm_bias_relu_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), out, M, N, K,
                              dtype_word(E4M3, F32, BF16), opts=opts)
        torch.cuda.synchronize()
        assert np.array_equal(down(out, BF16), oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, F32, BF16).out)
    # the gate and the residual with two K rows (two-stage ring beside the staged Y)
    p = gen.integer_problem(M, N, K, F16, F16, seed=M + 4, gate=True)
    out, _ = run_fused(p, M, N, K, F16, F16, F16, gate=True, opts=dict(opts, y_blocks=1))
    assert np.array_equal(down(out, F16), oracle_run(p, M, N, K, F16, F16, F16, gate=True).out)


@pytest.mark.parametrize("M,N,K,max_ctas", [(300, 520, 200, 0), (700, 1800, 200, 44), (513, 1288, 64, 12),
                                           (1000, 2056, 504, 0)])
def test_staged_y_two_blocks_single_cta_integer_bit_exact(M, N, K, max_ctas):
    # Two staged Y blocks per epilogue warp on single CTAs (Y two work items ahead, a two-stage
    # ring), with the bias added by the epilogue, written into tensor memory, or by the MMA form
    # (which then falls back to tensor memory: its tiles have no room beside two Y blocks)
    for bias_init, bias_mma in ((2, 0), (1, 1), (1, 2)):
        opts = {"path": fg.PATH_TC, "cta_pair": 1, "max_ctas": max_ctas, "y_blocks": 2,
                "bias_init": bias_init, "bias_mma": bias_mma}
        for ab in (F16, BF16):
            p = gen.integer_problem(M, N, K, ab, ab, seed=M + K + ab, gate=True)
            plan = fg.fgemm_plan(up(p.A, ab), up(p.B, ab), up(p.bias, ab), up(p.Y, ab),
                                 torch.empty(M, N, dtype=torch_dtype(ab), device="cuda"), M, N, K,
                                 dtype_word(ab, ab, ab), gate=True, opts=opts)
            assert (plan["cluster"], plan["y_blocks"]) == (1, 2)
            assert plan["bias_init"] == (0 if bias_init == 2 else 1)
            out, path = run_fused(p, M, N, K, ab, ab, ab, gate=True, opts=opts)
            assert path == fg.PATH_TC
            assert _same_values(down(out, ab), oracle_run(p, M, N, K, ab, ab, ab, gate=True).out, ab)
            res = torch.empty(M, N, dtype=torch_dtype(ab), device="cuda")
            fg.fgemm_bias_residual_relu_ex(up(p.A, ab), up(p.B, ab), up(p.bias, ab), up(p.Y, ab),
                                           res, M, N, K, dtype_word(ab, ab, ab), opts=opts)
            torch.cuda.synchronize()
            ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ab)
            assert _same_values(down(res, ab), ref.out, ab)


@pytest.mark.parametrize("M,N,K,max_ctas", [(300, 520, 200, 0), (700, 1800, 200, 44), (513, 1288, 64, 12),
                                           (1000, 2056, 504, 0), (129, 264, 8, 0)])
def test_sixteen_epilogue_warps_integer_bit_exact(M, N, K, max_ctas):
    # Sixteen epilogue warps on single CTAs (four per TMEM lane quadrant, 64 columns each, one
    # staged Y block per warp) for the gate and the residual, with the bias added after the sum,
    # written into tensor memory, or set by the extra MMA; tail pieces and the narrowed last tile.
    for bias_init, bias_mma in ((2, 0), (1, 1), (1, 2)):
        opts = {"path": fg.PATH_TC, "cta_pair": 1, "max_ctas": max_ctas, "epi_warps": 16,
                "bias_init": bias_init, "bias_mma": bias_mma}
        for ab in (F16, BF16):
            p = gen.integer_problem(M, N, K, ab, ab, seed=M + K + 3 * ab, gate=True)
            plan = fg.fgemm_plan(up(p.A, ab), up(p.B, ab), up(p.bias, ab), up(p.Y, ab),
                                 torch.empty(M, N, dtype=torch_dtype(ab), device="cuda"), M, N, K,
                                 dtype_word(ab, ab, ab), gate=True, opts=opts)
            assert (plan["cluster"], plan["epi_warps"]) == (1, 16)
            out, path = run_fused(p, M, N, K, ab, ab, ab, gate=True, opts=opts)
            assert path == fg.PATH_TC
            assert _same_values(down(out, ab), oracle_run(p, M, N, K, ab, ab, ab, gate=True).out, ab)
            res = torch.empty(M, N, dtype=torch_dtype(ab), device="cuda")
            fg.fgemm_bias_residual_relu_ex(up(p.A, ab), up(p.B, ab), up(p.bias, ab), up(p.Y, ab),
                                           res, M, N, K, dtype_word(ab, ab, ab), opts=opts)
            torch.cuda.synchronize()
            ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ab)
            assert _same_values(down(res, ab), ref.out, ab)
    # fp8 operands with a 16-bit Y
    p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + 11, gate=True, y_type=F16)
    if N % 16 == 0 and K % 16 == 0:
        out = torch.empty(M, N, dtype=torch.float16, device="cuda")
        fg.fgemm_addmm_gate_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), up(p.Y, F16), out, M, N,
                               K, dtype_word(E4M3, F32, F16, F16),
                               opts={"cta_pair": 1, "max_ctas": max_ctas, "epi_warps": 16})
        torch.cuda.synchronize()
        ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, E4M3, F32, F16, y_type=F16)
        assert _same_values(down(out, F16), ref.out, F16)


def _same_values(got_bits, ref_bits, t):
    """Equal as numbers (-0 == +0), every element."""
    return np.array_equal(oracle.decode(got_bits, t), oracle.decode(ref_bits, t))


@pytest.mark.parametrize("M,N,K,opts", BIAS_INIT_CASES)
def test_bias_init_integer_exact(M, N, K, opts):
    # "Optimizing GEMM + Activation on CDNA4 with TLX", V4: the accumulator starts at the bias.
    # With integer inputs every partial sum is exact in either order, so each epilogue must match
    # the oracle (bias added once after the sum) exactly; covers tail pieces, the narrowed last
    # tile, one-K-block tiles and both CTA modes.  Values are compared, so that an exact zero may
    # carry either sign (the sign of a zero sum depends on the order of the terms).
    o = dict(opts or {}, bias_init=1, path=fg.PATH_TC)
    for gate in (False, True):
        p = gen.integer_problem(M, N, K, BF16, BF16, seed=M + N + K + gate, gate=gate)
        out, path = run_fused(p, M, N, K, BF16, BF16, BF16, gate=gate, opts=o)
        assert path == fg.PATH_TC
        assert _same_values(down(out, BF16), oracle_run(p, M, N, K, BF16, BF16, BF16, gate=gate).out, BF16)
    # fp32 bias and output
    p = gen.integer_problem(M, N, K, F16, F32, seed=M + 3)
    out, _ = run_fused(p, M, N, K, F16, F32, F32, opts=o)
    assert _same_values(down(out, F32), oracle_run(p, M, N, K, F16, F32, F32).out, F32)
    # residual add
    p = gen.integer_problem(M, N, K, F16, F16, seed=M + 5, gate=True)
    out = torch.empty(M, N, dtype=torch.float16, device="cuda")
    fg.fgemm_bias_residual_relu_ex(up(p.A, F16), up(p.B, F16), up(p.bias, F16), up(p.Y, F16), out,
                                   M, N, K, fg.F16, opts=o)
    torch.cuda.synchronize()
    ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, F16)
    assert _same_values(down(out, F16), ref.out, F16)
    # quantized fp8 output (N a multiple of 16)
    if N % 16 == 0:
        p = gen.integer_problem(M, N, K, BF16, F32, seed=M + 7)
        got, path = _run_quant(p, M, N, K, BF16, F32, 0.25, o)
        assert path == fg.PATH_TC
        assert _same_values(got, oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, BF16, F32, 0.25).out, E4M3)
    # fp8 operands (K and N multiples of 16)
    if N % 16 == 0 and K % 16 == 0:
        p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + 9)
        out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        fg.fgemm_bias_relu_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), out, M, N, K,
                              dtype_word(E4M3, F32, BF16), opts=o)
        torch.cuda.synchronize()
        assert _same_values(down(out, BF16),
                            oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, F32, BF16).out, BF16)


BIAS_MMA_CASES = [  # M, N, K, opts: single CTAs, CTA pairs with one Y block, tail pieces,
    # the narrowed last tile (N = 1288 = 5 x 256 + 8), one-K-block tiles
    (300, 520, 200, {"cta_pair": 1}), (700, 1800, 200, {"cta_pair": 1, "max_ctas": 44}),
    (513, 1288, 328, {"cta_pair": 2, "y_blocks": 1}), (700, 1800, 600, {"cta_pair": 2, "max_ctas": 20}),
    (129, 264, 8, {"cta_pair": 1}), (1000, 1288, 1024, None)]


@pytest.mark.parametrize("M,N,K,opts", BIAS_MMA_CASES)
def test_bias_mma_integer_exact(M, N, K, opts):
    # The bias-initialised accumulator set by one extra MMA (ones x the staged bias row) must give
    # the oracle's values exactly on integer inputs, as the form written by the epilogue does, for
    # the gate and the residual add with 16-bit bias of the operand type.
    o = dict(opts or {}, bias_init=1, bias_mma=2, path=fg.PATH_TC)
    for ab in (F16, BF16):
        for epi in ("gate", "residual"):
            p = gen.integer_problem(M, N, K, ab, ab, seed=M + N + K + ab, gate=True)
            A, B, bias, R = up(p.A, ab), up(p.B, ab), up(p.bias, ab), up(p.Y, ab)
            word = dtype_word(ab, ab, ab)
            plan = fg.fgemm_plan(A, B, bias, R, torch.empty(1, device="cuda"), M, N, K, word, opts=o,
                                 epilogue=fg.EPI_GATE if epi == "gate" else fg.EPI_RESIDUAL_RELU)
            assert plan["bias_init"] == 2, plan  # the MMA form runs
            outs = []
            for form in ({}, {"bias_mma": 1}, {"bias_mma": 0}):
                out = torch.full((M, N), float("nan"), dtype=torch_dtype(ab), device="cuda")
                if epi == "gate":
                    fg.fgemm_addmm_gate_ex(A, B, bias, R, out, M, N, K, word, opts=dict(o, **form))
                else:
                    fg.fgemm_bias_residual_relu_ex(A, B, bias, R, out, M, N, K, word, opts=dict(o, **form))
                torch.cuda.synchronize()
                outs.append(down(out, ab))
            if epi == "gate":
                ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ab).out
            else:
                ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ab).out
            for got in outs:
                assert _same_values(got, ref, ab), (epi, ab)


def test_bias_init_default_on_short_k_only():
    # automatic choice: bias first for K <= 1024, after the sum above; forcing it off (2) gives the
    # after-the-sum order at any K, which on integer inputs is the same value
    M, N = 300, 520
    for K, default_bias_first in ((200, True), (1096, False)):
        p = gen.integer_problem(M, N, K, BF16, BF16, seed=K)
        auto, _ = run_fused(p, M, N, K, BF16, BF16, BF16, opts={"path": fg.PATH_TC})
        on, _ = run_fused(p, M, N, K, BF16, BF16, BF16, opts={"path": fg.PATH_TC, "bias_init": 1})
        off, _ = run_fused(p, M, N, K, BF16, BF16, BF16, opts={"path": fg.PATH_TC, "bias_init": 2})
        ref = oracle_run(p, M, N, K, BF16, BF16, BF16).out
        for x in (auto, on, off):
            assert _same_values(down(x, BF16), ref, BF16)
        assert torch.equal(auto, on if default_bias_first else off)


@pytest.mark.parametrize("gate", [False, True])
def test_bias_init_random_tolerance(gate):
    # random inputs: bias first changes only the rounding order of the fp32 sum
    M, N, K = 513, 1288, 1024
    p = gen.random_problem(M, N, K, F16, F16, seed=18, gate=gate)
    out, path = run_fused(p, M, N, K, F16, F16, F16, gate=gate, opts={"bias_init": 1})
    assert path == fg.PATH_TC
    ref = oracle_run(p, M, N, K, F16, F16, F16, gate=gate)
    check_close(down(out, F16), ref, K, F16, Y64=oracle.decode(p.Y, F16) if gate else None,
                bias64=oracle.decode(p.bias, F16), what="bias-init")


def test_bias_init_full_size_gate_sampled_rows():
    w = gen.WORKLOADS["glu_gate_1024x21568x4096"]
    x = gen.make(w)
    out, path = run_fused(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type, gate=True,
                          opts={"bias_init": 1})
    assert path == fg.PATH_TC
    rows = sample_rows(w.M)
    ref = oracle_run(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type, gate=True, rows=rows)
    check_close(down(out, w.out_type)[rows], ref, w.K, w.out_type,
                Y64=oracle.decode(x.Y[rows], w.y_type), bias64=oracle.decode(x.bias, w.bias_type),
                what="gate bias-init")


# ----------------------------------------------------------- float tolerance --

def test_small_ragged_workload_tc_and_generic():
    w = gen.WORKLOADS["ragged_200x136x72"]
    x = gen.make(w)
    ref = oracle_run(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type)
    b64 = oracle.decode(x.bias, w.bias_type)
    for path in (fg.PATH_TC, fg.PATH_GENERIC):
        out, taken = run_fused(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type, opts={"path": path})
        assert taken == path
        check_close(down(out, w.out_type), ref, w.K, w.out_type, bias64=b64, what=f"path {path}")


@pytest.mark.parametrize("gate", [False, True])
def test_random_tc_unit_scale(gate):
    # unit-scale inputs: the GEMM term dominates the bias, so the tolerance is sensitive to it
    M, N, K = 333, 776, 1024
    p = gen.random_problem(M, N, K, BF16, BF16, seed=9, scale=K ** -0.25, gate=gate)
    out, path = run_fused(p, M, N, K, BF16, BF16, BF16, gate=gate)
    assert path == fg.PATH_TC
    ref = oracle_run(p, M, N, K, BF16, BF16, BF16, gate=gate)
    check_close(down(out, BF16), ref, K, BF16, Y64=oracle.decode(p.Y, BF16) if gate else None,
                bias64=oracle.decode(p.bias, BF16), what="unit-scale")


# ----------------------------------------------------- coverage and ordering --

@pytest.mark.parametrize("M,N,K", [(200, 136, 72), (513, 776, 64)])
def test_tile_coverage_sentinel_and_guards(M, N, K):
    # every output element written once, nothing written outside out ("I3 ...": every tile exactly
    # once; "Triton: ReLU ...", "Mask discipline": the store mask protects memory past the end)
    p = gen.random_problem(M, N, K, F16, F16, seed=2)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.float16, device="cuda")
    out = buf[guard:guard + M * N].view(M, N)
    _, path = run_fused(p, M, N, K, F16, F16, F16, out=out)
    assert path == fg.PATH_TC
    b = buf.cpu()
    assert torch.isnan(b[:guard]).all() and torch.isnan(b[guard + M * N:]).all()
    assert not torch.isnan(b[guard:guard + M * N]).any()


@pytest.mark.parametrize("pair", [1, 2])
def test_grouping_and_grid_do_not_change_results(pair):
    M, N, K = 700, 1800, 128
    p = gen.random_problem(M, N, K, BF16, BF16, seed=4)
    base, _ = run_fused(p, M, N, K, BF16, BF16, BF16, opts={"cta_pair": pair})
    for opts in ({"group_m": 1}, {"group_m": 4}, {"group_m": 3, "max_ctas": 7}, {"max_ctas": 2},
                 {"raster": 1}, {"raster": 1, "group_m": 3}):
        out, _ = run_fused(p, M, N, K, BF16, BF16, BF16, opts=dict(opts, cta_pair=pair))
        assert torch.equal(out, base), opts


@pytest.mark.parametrize("pair,max_ctas", [(1, 20), (1, 35), (1, 44), (2, 12), (2, 20), (2, 40)])
def test_tail_round_pieces_integer_bit_exact(pair, max_ctas):
    # The last partial round of the persistent grid is cut into 128- or 64-column pieces; a grid
    # cap chosen per case makes 2 or 4 pieces per tail tile, on ragged M, N and K.
    M, N, K = 700, 1800, 200
    for gate in (False, True):
        p = gen.integer_problem(M, N, K, BF16, BF16, seed=max_ctas, gate=gate)
        out, path = run_fused(p, M, N, K, BF16, BF16, BF16, gate=gate,
                              opts={"cta_pair": pair, "max_ctas": max_ctas})
        assert path == fg.PATH_TC
        ref = oracle_run(p, M, N, K, BF16, BF16, BF16, gate=gate)
        assert np.array_equal(down(out, BF16), ref.out)
        whole, _ = run_fused(p, M, N, K, BF16, BF16, BF16, gate=gate,
                             opts={"cta_pair": pair, "max_ctas": max_ctas, "tail_split": 1})
        assert torch.equal(whole, out)


def test_pair_and_single_cta_agree():
    M, N, K = 1000, 2056, 512
    p = gen.random_problem(M, N, K, F16, F16, seed=14)
    a, _ = run_fused(p, M, N, K, F16, F16, F16, opts={"cta_pair": 1})
    b, _ = run_fused(p, M, N, K, F16, F16, F16, opts={"cta_pair": 2})
    ref = oracle_run(p, M, N, K, F16, F16, F16)
    for x in (a, b):
        check_close(down(x, F16), ref, K, F16, bias64=oracle.decode(p.bias, F16), what="pair/single")


SKINNY_FP8_SHAPES = [(1, 144, 128, 1), (5, 272, 512, 3), (16, 1040, 2048, 4), (33, 400, 256, 2),
                     (64, 144, 32, 4), (100, 528, 1024, 8), (128, 1040, 512, 2)]


@pytest.mark.parametrize("M,N,K,split", SKINNY_FP8_SHAPES)
@pytest.mark.parametrize("tiles", [1, 2])
def test_skinny_fp8_integer_bit_exact(M, N, K, split, tiles):
    # fp8 e4m3 operands on the swap-AB kernel (kind::f8f6f4, 128 K elements per stage): bias +
    # ReLU, the gate with a 16-bit Y, and the quantized output; (64, 144, 32, 4) leaves three of
    # the four CTAs of each cluster without a K block
    o = {"split_k": split, "skinny_tiles": tiles}
    for bt, ot in ((F32, BF16), (BF16, F32)):
        p = gen.integer_problem(M, N, K, E4M3, bt, seed=M + N + K + split)
        out = torch.empty(M, N, dtype=torch_dtype(ot), device="cuda")
        path = fg.fgemm_bias_relu_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, bt), out, M, N, K,
                                     dtype_word(E4M3, bt, ot), opts=o)
        torch.cuda.synchronize()
        assert path == fg.PATH_SKINNY
        assert _same_values(down(out, ot), oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, bt, ot).out, ot)
    p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + K, gate=True, y_type=F16)
    out = torch.empty(M, N, dtype=torch.float16, device="cuda")
    fg.fgemm_addmm_gate_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), up(p.Y, F16), out, M, N,
                           K, dtype_word(E4M3, F32, F16, F16), opts=o)
    torch.cuda.synchronize()
    ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, E4M3, F32, F16, y_type=F16)
    assert _same_values(down(out, F16), ref.out, F16)
    p = gen.integer_problem(M, N, K, E4M3, F32, seed=M + 7)
    out = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    fg.fgemm_bias_relu_quant_ex(up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32), out, M, N, K,
                                fg.E4M3 | fg.BIAS_F32 | fg.OUT_E4M3, 0.25, opts=o)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, E4M3, F32, 0.25).out)


# -------------------------------------------------------------- unfused chain --

@pytest.mark.parametrize("inter_f32", [0, 1])
@pytest.mark.parametrize("gate", [False, True])
def test_unfused_chain_matches_oracle(inter_f32, gate):
    M, N, K = 257, 520, 192
    p = gen.random_problem(M, N, K, F16, F16, seed=8, gate=gate)
    ref = oracle_run(p, M, N, K, F16, F16, F16, gate=gate)
    ws_bytes = fg.fgemm_unfused_workspace_bytes(M, N, fg.F16, inter_f32)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(M, N, dtype=torch.float16, device="cuda")
    args = (up(p.A, F16), up(p.B, F16), up(p.bias, F16))
    if gate:
        fg.fgemm_unfused_addmm_gate(*args, up(p.Y, F16), out, M, N, K, fg.F16, ws, ws_bytes, inter_f32)
    else:
        fg.fgemm_unfused_bias_relu(*args, out, M, N, K, fg.F16, ws, ws_bytes, inter_f32)
    torch.cuda.synchronize()
    got = oracle.decode(down(out, F16), F16)
    want = oracle.decode(ref.out, F16)
    from gpu_util import tolerance
    assert float(np.abs(got - want).max()) <= tolerance(K, want, F16)


# ------------------------------------------------------------ full-size sampled --

FULL = ["square_4096", "glu_gate_1024x21568x4096", "glu_gate_fp8_1024x21568x4096",
        "ffn_up_8192x14336x4096", "ffn_up_fp8_8192x14336x4096",
        "square_fp8_4096", "skinny_M1_8192",
        "skinny_M16_8192", "skinny_M64_8192", "skinny_M128_8192", "skinny_fp8_M1_8192",
        "skinny_fp8_M16_8192", "skinny_fp8_M64_8192", "skinny_fp8_M128_8192", "glu_gate_1024x21568x256",
        "glu_gate_1024x21568x512", "glu_gate_1024x21568x1024", "ragged_200x136x72"]

_made = {}


def made(name):
    """The workload's seeded inputs, drawn once per test session (the last one kept)."""
    if name not in _made:
        _made.clear()
        _made[name] = gen.make(gen.WORKLOADS[name])
    return _made[name]


def launch_opts(dev_in, w, launch):
    """Options of the launch under test: `bench` is the launch bench.py times (library defaults,
    which cut the tiles of the persistent grid's last partial round into column pieces);
    `whole_tiles` keeps those tiles whole.  None when `whole_tiles` is the same launch."""
    if launch == "bench":
        return {}
    A, B, bias, Y, out = dev_in
    plan = fg.fgemm_plan(A, B, bias, Y, out, w.M, w.N, w.K,
                         dtype_word(w.ab_type, w.bias_type, w.out_type, w.y_type),
                         gate=Y is not None)
    if plan["path"] != fg.PATH_TC or plan["tail_split"] == 1:
        return None
    return {"tail_split": 1}


_oracle_rows = {}


def oracle_rows(name, x, w, rows):
    key = (name, tuple(rows[:4]), len(rows))
    if key not in _oracle_rows:
        _oracle_rows.clear()
        _oracle_rows[key] = oracle_run(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type,
                                       gate=w.epilogue == "gate", rows=rows, y_type=w.y_type)
    return _oracle_rows[key]


FULL_CASES = [(n, launch) for n in FULL for launch in ("bench", "whole_tiles")]


def run_full(x, w, launch, what):
    """One full-size launch into a NaN-prefilled output with guard bands; checks that every
    element was written and nothing outside it.  Returns the output, or None when the launch is
    the same as `bench`."""
    gate = w.epilogue == "gate"
    out, buf = guarded_out(w.M, w.N, w.out_type)
    dev_in = (up(x.A, w.ab_type), up(x.B, w.ab_type), up(x.bias, w.bias_type),
              up(x.Y, w.y_type) if gate else None, out)
    opts = launch_opts(dev_in, w, launch)
    if opts is None:
        return None
    A, B, bias, Y, _ = dev_in
    word = dtype_word(w.ab_type, w.bias_type, w.out_type, w.y_type)
    if gate:
        fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, w.M, w.N, w.K, word, opts=opts or None)
    else:
        fg.fgemm_bias_relu_ex(A, B, bias, out, w.M, w.N, w.K, word, opts=opts or None)
    torch.cuda.synchronize()
    check_guarded(buf, w.M, w.N, w.out_type, what=what)
    return out


@pytest.mark.parametrize("name,launch", FULL_CASES)
def test_full_size_workloads(name, launch):
    """Every configuration at its full size.  `bench`: the launch bench.py times; `whole_tiles`:
    the tiles of the persistent grid's last partial round kept whole instead of cut into column
    pieces (skipped where that is the same launch).  Every output element must be written and
    nothing outside the output (NaN-prefilled buffer with guard bands), and a stratified row
    sample (every epilogue warp's rows of every M tile, the ragged last tile) must match the
    oracle within the stated tolerance and the per-element forward-error bound."""
    w = gen.WORKLOADS[name]
    x = made(name)
    gate = w.epilogue == "gate"
    out = run_full(x, w, launch, f"{name}/{launch}")
    if out is None:
        pytest.skip("the tail round is not cut on this shape: the same launch as `bench`")
    rows = sample_rows(w.M)
    ref = oracle_rows(name, x, w, rows)
    got = down(out, w.out_type)[rows]
    Y64 = oracle.decode(x.Y[rows], w.y_type) if gate else None
    b64 = oracle.decode(x.bias, w.bias_type)
    check_close(got, ref, w.K, w.out_type, Y64=Y64, bias64=b64, what=f"{name}/{launch}")
    if launch == "bench":
        # negative control: an output that left out the GEMM term must fail the per-element bound
        fake = oracle.gemm_epilogue(x.A, x.B, x.bias, w.M, w.N, w.K, w.ab_type, w.bias_type,
                                    w.out_type, oracle.EPI_GATE if gate else oracle.EPI_RELU,
                                    Y=x.Y, rows=rows, mutant=oracle.MUT_DROP_GEMM, y_type=w.y_type)
        with pytest.raises(AssertionError):
            check_close(fake.out, ref, w.K, w.out_type, Y64=Y64, bias64=b64, what="bias-only control")


@pytest.mark.parametrize("name,launch", [("square_4096", "bench"), ("square_4096", "whole_tiles"),
                                         ("glu_gate_1024x21568x4096", "bench"),
                                         ("glu_gate_1024x21568x4096", "whole_tiles")])
def test_full_size_integer_every_element_bit_exact(name, launch):
    """The two gated configurations at full size on small-integer inputs (every partial sum exact
    in fp32, so the one rounding is the final one): every element of the output equals the oracle
    bit for bit, which shows every output tile written exactly once with its own tile's value, in
    the launch bench.py times and with whole tail tiles.  The gate takes values in [-1, 1] so
    that X + X * Y stays finite in fp16."""
    w = gen.WORKLOADS[name]
    gate = w.epilogue == "gate"
    lo, hi = (-1, 1) if gate else (-3, 3)
    key = ("int", name)
    if key not in _made:
        _made.clear()
        _made[key] = gen.integer_problem(w.M, w.N, w.K, w.ab_type, w.bias_type, seed=w.seed,
                                         lo=lo, hi=hi, gate=gate)
    x = _made[key]
    out = run_full(x, w, launch, f"{name}/{launch}")
    assert out is not None
    rkey = ("int-oracle", name)
    if rkey not in _oracle_rows:
        _oracle_rows.clear()
        _oracle_rows[rkey] = oracle_run(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type,
                                        gate=gate)
    want = _oracle_rows[rkey].out
    got = down(out, w.out_type)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")


def test_plan_matches_the_path_that_runs():
    cases = [(4096, 4096, 512, False, None), (1024, 21568, 256, True, None), (16, 8192, 1024, False, None),
             (700, 1800, 200, False, {"cta_pair": 1, "max_ctas": 44}), (3, 5, 7, False, None)]
    for M, N, K, gate, opts in cases:
        p = gen.random_problem(M, N, K, F16, F16, seed=1, gate=gate)
        A, B, bias, Y = up(p.A, F16), up(p.B, F16), up(p.bias, F16), up(p.Y, F16) if gate else None
        out = torch.empty(M, N, dtype=torch.float16, device="cuda")
        plan = fg.fgemm_plan(A, B, bias, Y, out, M, N, K, fg.F16, gate=gate, opts=opts)
        if gate:
            path = fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, fg.F16, opts=opts)
        else:
            path = fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, fg.F16, opts=opts)
        torch.cuda.synchronize()
        assert plan["path"] == path
        if path == fg.PATH_TC:
            assert plan["grid"] % plan["cluster"] == 0 and plan["grid"] > 0
            units = plan["grid"] // plan["cluster"]
            rem = plan["tiles"] % units
            assert plan["work_items"] == plan["tiles"] + rem * (plan["tail_split"] - 1) or \
                plan["tail_split"] == 1
    # the split of the 44-CTA single-CTA case: 48 tiles on 44 CTAs -> 4 tail tiles in 4 pieces
    p = gen.random_problem(700, 1800, 200, F16, F16, seed=1)
    plan = fg.fgemm_plan(up(p.A, F16), up(p.B, F16), up(p.bias, F16), None,
                         torch.empty(700, 1800, dtype=torch.float16, device="cuda"), 700, 1800, 200,
                         fg.F16, opts={"cta_pair": 1, "max_ctas": 44})
    assert (plan["tiles"], plan["grid"], plan["tail_split"], plan["work_items"]) == (48, 44, 4, 60)


def test_device_error_word_clear():
    assert fg.fgemm_device_status() == 0
