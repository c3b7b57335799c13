"""Seeded random shapes through every entry point on the path the library picks, against the
oracle.  Small-integer inputs keep every partial sum exact, so each output must equal the
oracle's (compared as values: a zero sum may carry either sign)."""
import numpy as np
import pytest

import oracle
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import BF16, E4M3, F16, F32, down, dtype_word, up

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gemm_epilogue_gb300.binding as fg  # noqa: E402

TORCH = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemm_epilogue_gb300 import build
    build.build()
    oracle.build()
    fg.lib()
    yield
    assert fg.fgemm_device_status() == 0


def _cases(n=48, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        aligned = rng.random() < 0.8
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 256)) * 8 if aligned else int(rng.integers(1, 2000))
        K = int(rng.integers(0, 80)) * 8 if aligned else int(rng.integers(0, 600))
        if rng.random() < 0.25:  # fp8 e4m3 operands: bias + ReLU or the quantized output
            epi = ["relu", "quant"][int(rng.integers(0, 2))]
            ab = E4M3
            bt = [F32, BF16][int(rng.integers(0, 2))]
            ot = [BF16, F32][int(rng.integers(0, 2))] if epi != "quant" else E4M3
        else:
            epi = ["relu", "gate", "resid", "quant"][int(rng.integers(0, 4))]
            ab = [F16, BF16][int(rng.integers(0, 2))]
            bt = [ab, F32][int(rng.integers(0, 2))]
            ot = [ab, F32][int(rng.integers(0, 2))] if epi != "quant" else E4M3
        if epi == "quant" and N % 16:
            N += 16 - N % 16 if aligned else 0
        out.append((i, M, N, K, epi, ab, bt, ot))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}x{c[3]}-{c[4]}")
def test_random_shapes_exact(case):
    i, M, N, K, epi, ab, bt, ot = case
    p = gen.integer_problem(M, N, K, ab, bt, seed=1000 + i, gate=epi in ("gate", "resid"))
    A = up(p.A, ab) if K else None
    B = up(p.B, ab) if K else None
    bias = up(p.bias, bt)
    Y = up(p.Y, ab) if epi in ("gate", "resid") else None
    if ot == E4M3:
        out = torch.empty(M, N, dtype=torch.uint8, device="cuda")
        fg.fgemm_bias_relu_quant(A, B, bias, out, M, N, K, dtype_word(ab, bt, E4M3), 0.25)
        torch.cuda.synchronize()
        ref = oracle.bias_relu_quant(p.A, p.B, p.bias, M, N, K, ab, bt, 0.25).out
        got = out.cpu().numpy()
    else:
        out = torch.empty(M, N, dtype=TORCH[ot], device="cuda")
        w = dtype_word(ab, bt, ot)
        if epi == "relu":
            fg.fgemm_bias_relu(A, B, bias, out, M, N, K, w)
            ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, ab, bt, ot).out
        elif epi == "gate":
            fg.fgemm_addmm_gate(A, B, bias, Y, out, M, N, K, w)
            ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, ab, bt, ot).out
        else:
            fg.fgemm_bias_residual_relu(A, B, bias, Y, out, M, N, K, w)
            ref = oracle.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, ab, bt, ot).out
        torch.cuda.synchronize()
        got = down(out, ot)
    g, r = oracle.decode(got, ot), oracle.decode(ref, ot)
    if not np.array_equal(g, r):
        bad = np.argwhere(g != r)
        pytest.fail(f"{len(bad)} mismatches, first at {bad[:5].tolist()}")
