"""GPU parity of the stream-K share-out of the tensor-core path's last round (fgemm_opts.stream_k):
bit-exact on integer inputs (every partial sum is exact in fp32, so the order in which the runs'
sums are added cannot show), within the tolerance on random inputs, the same bits on every call
with the same plan, every element written once, and the workspace's flags left at zero."""

import numpy as np
import pytest

import oracle
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import BF16, E4M3, F16, F32, check_close, down, dtype_word, sample_rows, up

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gemm_epilogue_gb300.binding as fg  # noqa: E402

TORCH_OF = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemm_epilogue_gb300 import build
    build.build()
    oracle.build()
    fg.lib()
    yield
    assert fg.fgemm_device_status() == 0


@pytest.fixture(scope="module")
def ws():
    # zero-filled once; every call that completes leaves the flag words zero again
    return torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")


def sk(ws, **kw):
    return dict(kw, stream_k=1, workspace=ws.data_ptr(), workspace_bytes=ws.numel())


def flags_clear(ws):
    return int(ws[:fg.SK_FLAG_BYTES].count_nonzero()) == 0


def run(p, M, N, K, ab, bt, ot, opts, gate=False, out=None):
    A, B, bias = up(p.A, ab), up(p.B, ab), up(p.bias, bt)
    Y = up(p.Y, ab) if gate else None
    if out is None:
        out = torch.empty(M, N, dtype=TORCH_OF[ot], device="cuda")
    w = dtype_word(ab, bt, ot)
    plan = fg.fgemm_plan(A, B, bias, Y, out, M, N, K, w, gate=gate, opts=opts)
    if gate:
        path = fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, w, opts=opts)
    else:
        path = fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, w, opts=opts)
    torch.cuda.synchronize()
    assert path == fg.PATH_TC
    return out, plan


# Ragged in M, N and K against the tiles: on pairs 3 x 8 tiles of 256 x 256 and K = 2048 = 16 K
# blocks of 128; on single CTAs 6 x 8 tiles of 128 x 256 and K = 1096 = 17 whole K blocks of 64
# and a partial one.  N = 1800 narrows the last column of tiles.  The grid caps make 2 to 8 tiles
# in the last round, shared out over 5 to 20 units.
CASES = [(2, 10), (2, 14), (2, 22), (1, 7), (1, 10), (1, 20)]


@pytest.mark.parametrize("pair,max_ctas", CASES)
def test_stream_k_integer_bit_exact(ws, pair, max_ctas):
    M, N = 700, 1800
    K = 2048 if pair == 2 else 1096
    for gate, ot in ((False, BF16), (False, F32), (True, F32)):
        p = gen.integer_problem(M, N, K, BF16, BF16, seed=max_ctas + K, gate=gate)
        out, plan = run(p, M, N, K, BF16, BF16, ot, sk(ws, cta_pair=pair, max_ctas=max_ctas),
                        gate=gate)
        assert plan["sk_tiles"] > 0
        ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, BF16, BF16, ot) if gate else \
            oracle.bias_relu(p.A, p.B, p.bias, M, N, K, BF16, BF16, ot)
        got = down(out, ot)
        if not np.array_equal(got, ref.out):
            bad = np.argwhere(got != ref.out)
            pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")
        assert flags_clear(ws)


# The gate and the residual with 16-bit outputs stage Y (or R) through shared memory: on pairs one
# 4 KB chunk at a time (K = 2048) or a whole block a work item ahead (K = 1024, one K row per
# stage, 16 K blocks), on single CTAs a block ahead (K = 1096).
STAGED = [(2, 10, 2048), (2, 14, 1024), (1, 10, 1096)]


@pytest.mark.parametrize("pair,max_ctas,K", STAGED)
def test_stream_k_staged_second_operand_bit_exact(ws, pair, max_ctas, K):
    M, N = 700, 1800
    opts = sk(ws, cta_pair=pair, max_ctas=max_ctas)
    for ab in (F16, BF16):
        p = gen.integer_problem(M, N, K, ab, ab, seed=K + max_ctas, gate=True)
        out, plan = run(p, M, N, K, ab, ab, ab, opts, gate=True)
        assert plan["sk_tiles"] > 0
        ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ab)
        assert np.array_equal(down(out, ab), ref.out)
        # the residual add stages R the same way
        out = torch.empty(M, N, dtype=TORCH_OF[ab], device="cuda")
        path = fg.fgemm_bias_residual_relu_ex(up(p.A, ab), up(p.B, ab), up(p.bias, ab), up(p.Y, ab),
                                              out, M, N, K, dtype_word(ab, ab, ab), opts=opts)
        torch.cuda.synchronize()
        assert path == fg.PATH_TC
        ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, ab, ab, ab)
        assert np.array_equal(down(out, ab), ref.out)
        assert flags_clear(ws)


def test_stream_k_quantized_output_bit_exact(ws):
    M, N, K = 700, 1808, 2048
    p = gen.integer_problem(M, N, K, BF16, F32, seed=3)
    out = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    w = fg.BF16 | fg.BIAS_F32 | fg.OUT_E4M3
    opts = sk(ws, cta_pair=2, max_ctas=10)
    assert fg.fgemm_plan(up(p.A, BF16), up(p.B, BF16), up(p.bias, F32), None, out, M, N, K, w,
                         opts=opts, epilogue=fg.EPI_RELU_QUANT)["sk_tiles"] > 0
    path = fg.fgemm_bias_relu_quant_ex(up(p.A, BF16), up(p.B, BF16), up(p.bias, F32), out, M, N, K,
                                       w, 0.125, opts=opts)
    torch.cuda.synchronize()
    assert path == fg.PATH_TC
    ref = oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, BF16, F32, 0.125)
    assert np.array_equal(out.cpu().numpy(), ref.out)
    assert flags_clear(ws)


def test_stream_k_fp8_operands_bit_exact(ws):
    # fp8 operands on pairs: two 128-element K rows per stage, K = 4096 is 16 K blocks
    M, N, K = 700, 1808, 4096
    p = gen.integer_problem(M, N, K, E4M3, F32, seed=5)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w = dtype_word(E4M3, F32, BF16)
    opts = sk(ws, max_ctas=10)
    A, B, bias = up(p.A, E4M3), up(p.B, E4M3), up(p.bias, F32)
    assert fg.fgemm_plan(A, B, bias, None, out, M, N, K, w, opts=opts)["sk_tiles"] > 0
    assert fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, w, opts=opts) == fg.PATH_TC
    torch.cuda.synchronize()
    ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, E4M3, F32, BF16)
    assert np.array_equal(down(out, BF16), ref.out)
    assert flags_clear(ws)


@pytest.mark.parametrize("pair,max_ctas", [(2, 14), (1, 20)])
def test_stream_k_random_tolerance_deterministic_and_covering(ws, pair, max_ctas):
    M, N = 700, 1800
    K = 2048 if pair == 2 else 1096
    p = gen.random_problem(M, N, K, BF16, BF16, seed=11)
    opts = sk(ws, cta_pair=pair, max_ctas=max_ctas)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out, plan = run(p, M, N, K, BF16, BF16, BF16, opts, out=buf[guard:guard + M * N].view(M, N))
    assert plan["sk_tiles"] > 0
    b = buf.cpu()
    assert torch.isnan(b[:guard]).all() and torch.isnan(b[guard + M * N:]).all()
    assert not torch.isnan(b[guard:guard + M * N]).any()
    ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, BF16, BF16, BF16)
    check_close(down(out, BF16), ref, K, BF16, bias64=oracle.decode(p.bias, BF16), what="stream-K")
    # the same plan gives the same bits, call after call
    for _ in range(3):
        again, _ = run(p, M, N, K, BF16, BF16, BF16, opts)
        assert torch.equal(again, out)
    assert flags_clear(ws)


@pytest.mark.parametrize("name", ["square_4096", "glu_gate_1024x21568x4096"])
def test_full_size_stream_k_sampled_rows(ws, name):
    w = gen.WORKLOADS[name]
    x = gen.make(w)
    opts = {"workspace": ws.data_ptr(), "workspace_bytes": ws.numel()}  # automatic mode
    gate = w.epilogue == "gate"
    out, plan = run(x, w.M, w.N, w.K, w.ab_type, w.bias_type, w.out_type, opts, gate=gate)
    assert plan["sk_tiles"] > 0
    rows = sample_rows(w.M)
    if gate:
        ref = oracle.addmm_gate(x.A, x.B, x.bias, x.Y, w.M, w.N, w.K, w.ab_type, w.bias_type,
                                w.out_type, rows=rows)
    else:
        ref = oracle.bias_relu(x.A, x.B, x.bias, w.M, w.N, w.K, w.ab_type, w.bias_type,
                               w.out_type, rows=rows)
    check_close(down(out, w.out_type)[rows], ref, w.K, w.out_type,
                Y64=oracle.decode(x.Y[rows], w.ab_type) if gate else None,
                bias64=oracle.decode(x.bias, w.bias_type), what=name + " stream-K")
    assert flags_clear(ws)
