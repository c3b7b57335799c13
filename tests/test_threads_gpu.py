"""First calls from several host threads at once: the library's per-device state (the
shared-memory opt-in of each kernel instance, the cached count of resident CTA pairs, the device
table, the no-allocation entry's address lookup) is set on first use and must tolerate threads
racing to set it.  Run in a fresh process, so that these really are the first calls."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import numpy as np, torch
import oracle
import gemm_epilogue_gb300.binding as fg
from gemm_epilogue_gb300 import inputs as gen
from gpu_util import F16, BF16, up, down, dtype_word
torch.cuda.init()
# shapes that take different kernel instances: CTA pairs, single CTAs, the skinny kernel, the
# gate with staged Y, the CUDA-core path, and the no-allocation entry
CASES = [(300, 520, 1096, "relu", BF16), (300, 520, 200, "relu", F16), (16, 1032, 512, "relu", BF16),
         (513, 1288, 328, "gate", F16), (7, 44, 9, "relu", F16), (129, 264, 72, "noalloc", F16)]
results = [None] * len(CASES)
barrier = threading.Barrier(len(CASES))

def run(i):
    M, N, K, epi, t = CASES[i]
    p = gen.integer_problem(M, N, K, t, t, seed=i, gate=epi == "gate")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A, B, bias = up(p.A, t), up(p.B, t), up(p.bias, t)
        Y = up(p.Y, t) if epi == "gate" else None
        out = torch.empty(M, N, dtype=torch.float16 if t == F16 else torch.bfloat16, device="cuda")
    s.synchronize()
    barrier.wait()  # every thread makes its first library call at the same moment
    w = dtype_word(t, t, t)
    if epi == "gate":
        fg.fgemm_addmm_gate_ex(A, B, bias, Y, out, M, N, K, w, s.cuda_stream)
        ref = oracle.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, t, t, t).out
    elif epi == "noalloc":
        fg.fgemm_unfused_bias_relu_noalloc(A, B, bias, out, M, N, K, w, 0, s.cuda_stream)
        ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, t, t, t).out
    else:
        fg.fgemm_bias_relu_ex(A, B, bias, out, M, N, K, w, s.cuda_stream)
        ref = oracle.bias_relu(p.A, p.B, p.bias, M, N, K, t, t, t).out
    s.synchronize()
    got = oracle.decode(down(out, t), t)
    results[i] = bool(np.array_equal(got, oracle.decode(ref, t)))

threads = [threading.Thread(target=run, args=(i,)) for i in range(len(CASES))]
for th in threads: th.start()
for th in threads: th.join()
assert fg.fgemm_device_status() == 0
print("RESULTS", results)
sys.exit(0 if all(results) else 1)
"""


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemm_epilogue_gb300 import build
    import oracle
    build.build()
    oracle.build()


def test_first_calls_from_several_threads_at_once():
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "RESULTS [True, True, True, True, True, True]" in r.stdout
