"""Failure detection on the GPU without faulting it: every barrier wait in the tensor-core and
skinny kernels is bounded.  A diagnostic option makes the first CTA announce a stage whose loads
it never issues (a barrier that nothing completes); the wait must expire after timeout_ms, the
kernel must drain and exit, fgemm_device_status must report FGEMM_ERR_TIMEOUT, and the context
must stay usable for the next call."""
import pytest

import oracle
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import BF16, check_close, down, up

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import gemm_epilogue_gb300.binding as fg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemm_epilogue_gb300 import build
    build.build()
    fg.lib()
    assert fg.fgemm_device_status() == 0


CASES = [  # (M, N, K, opts that select the path)
    (700, 1800, 512, {"cta_pair": 1}),
    (700, 1800, 512, {"cta_pair": 2}),
    (16, 2048, 2048, {"path": 2}),
]


@pytest.mark.parametrize("M,N,K,sel", CASES)
def test_stalled_wait_times_out_and_the_context_survives(M, N, K, sel):
    p = gen.random_problem(M, N, K, BF16, BF16, seed=3)
    A, B, bias = up(p.A, BF16), up(p.B, BF16), up(p.bias, BF16)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    path = fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, fg.BF16,
                                 opts=dict(sel, inject_stall=1, timeout_ms=50))
    code = fg.fgemm_device_status()            # synchronises: the kernel has ended
    assert code & 0xFF == fg.ERR_TIMEOUT, hex(code)
    assert fg.fgemm_device_status() == 0       # read-and-clear
    # the same call without the stall is correct afterwards
    path2 = fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, fg.BF16, opts=sel)
    assert path2 == path
    torch.cuda.synchronize()
    ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, BF16, BF16, BF16)
    check_close(down(out, BF16), ref, K, BF16, bias64=oracle.decode(p.bias, BF16), what="after stall")
    assert fg.fgemm_device_status() == 0
