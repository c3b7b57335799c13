"""Programmatic dependent launch (fgemm_opts.pdl, on by default): a call's set-up may overlap the
previous kernel, but its first global-memory access waits for that kernel to complete.  A chain in
which each call reads the previous call's output must therefore give the oracle's result, launched
one by one and from a captured CUDA graph."""
import numpy as np
import pytest

import oracle
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import BF16, down, up

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


# tensor-core pairs (a short and a long K loop), tensor-core single CTAs, skinny
CASES = [(700, 1800, 1024, {"cta_pair": 2}), (520, 1032, 2112, {}), (300, 520, 200, {"cta_pair": 1}),
         (16, 1032, 512, {})]


@pytest.mark.parametrize("M,N,K,sel", CASES)
@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("pdl", [1, 0])
def test_chain_reads_the_previous_output(M, N, K, sel, graph, pdl):
    # out1 = ReLU(A B + bias); out2 = X + X * out1 with X = A B + bias: the second call's Y is
    # the first call's output, written just before it starts.  Integer inputs keep both exact.
    p = gen.integer_problem(M, N, K, BF16, BF16, seed=M + K, lo=-1, hi=1)
    A, B, bias = up(p.A, BF16), up(p.B, BF16), up(p.bias, BF16)
    out1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    opts = dict(sel, pdl=pdl)  # 0: the automatic choice, which is on
    stream = torch.cuda.Stream()

    def chain():
        s = stream.cuda_stream
        fg.fgemm_bias_relu_ex(A, B, bias, out1, M, N, K, fg.BF16, s, opts)
        fg.fgemm_addmm_gate_ex(A, B, bias, out1, out2, M, N, K, fg.BF16, s, opts)

    if graph:
        chain()  # first calls outside capture (device set-up)
        torch.cuda.synchronize()
        out1.fill_(float("nan"))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            chain()
        g.replay()
    else:
        with torch.cuda.stream(stream):
            chain()
    torch.cuda.synchronize()
    ref1 = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, BF16, BF16, BF16)
    assert np.array_equal(down(out1, BF16), ref1.out)
    ref2 = oracle.addmm_gate(p.A, p.B, p.bias, ref1.out, M, N, K, BF16, BF16, BF16)
    assert np.array_equal(down(out2, BF16), ref2.out)
    assert fg.fgemm_device_status() == 0
