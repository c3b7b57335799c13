"""fgemm_unfused_bias_relu_noalloc: the unfused bias + ReLU chain for callers that cannot
allocate device memory (its intermediate lives in an array the library reserves on each device).

Checked on two calls in a row against the existing entry point fgemm_unfused_bias_relu (given
a workspace from the caller) and against the CPU oracle, with the same tolerance as the other
parity tests.  This file is
collected last so that a run stopping at its first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import oracle
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import F16, BF16, down, tolerance, up

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


def _both(p, M, N, K, t, inter_f32):
    word = fg.F16 if t == F16 else fg.BF16
    tdt = torch.float16 if t == F16 else torch.bfloat16
    A, B, bias = up(p.A, t), up(p.B, t), up(p.bias, t)
    nbytes = fg.fgemm_unfused_workspace_bytes(M, N, word, inter_f32)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    want = torch.empty(M, N, dtype=tdt, device="cuda")
    got = torch.empty(M, N, dtype=tdt, device="cuda")
    fg.fgemm_unfused_bias_relu(A, B, bias, want, M, N, K, word, ws, nbytes, inter_f32)
    fg.fgemm_unfused_bias_relu_noalloc(A, B, bias, got, M, N, K, word, inter_f32)
    torch.cuda.synchronize()
    return down(got, t), down(want, t)


def test_noalloc_matches_the_workspace_entry_on_two_calls_in_a_row():
    # the second call uses another shape, type and seed, so anything the first call left in the
    # shared array would show up as a mismatch
    cases = [(300, 520, 200, F16, 0, 31), (129, 264, 72, BF16, 1, 32)]
    for M, N, K, t, inter_f32, seed in cases:
        p = gen.random_problem(M, N, K, t, t, seed=seed)
        got, want = _both(p, M, N, K, t, inter_f32)
        g64, w64 = oracle.decode(got, t), oracle.decode(want, t)
        assert np.all(np.isfinite(g64))
        assert float(np.abs(g64 - w64).max()) <= tolerance(K, w64, t)
        # and against the oracle (fp64 sum, bias and ReLU after it, one rounding), so that a fault
        # shared by both CUDA chains cannot pass
        ref = oracle.decode(oracle.bias_relu(p.A, p.B, p.bias, M, N, K, t, t, t).out, t)
        assert float(np.abs(g64 - ref).max()) <= tolerance(K, ref, t)
    assert fg.fgemm_device_status() == 0


def test_noalloc_rejects_a_problem_larger_than_its_array():
    # 4096 x 4096 fp16 intermediate = 32 MiB > the 16 MiB array: refused, nothing runs
    M, N, K = 4096, 4096, 8
    A = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.float16, device="cuda")
    bias = torch.zeros(N, dtype=torch.float16, device="cuda")
    out = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda")
    assert fg.fgemm_unfused_workspace_bytes(M, N, fg.F16, 0) > fg.NOALLOC_SCRATCH_BYTES
    st = fg.call_status("fgemm_unfused_bias_relu_noalloc", A.data_ptr(), B.data_ptr(),
                        bias.data_ptr(), out.data_ptr(), M, N, K, fg.F16, 0, None)
    assert st == fg.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
