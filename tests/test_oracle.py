"""Pins for the fp64 oracle: what the pages print, closed forms, library
routines on special cases, exact brute force, and negative controls showing
each pin rejects a plausible mistake.  CPU only."""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import parse_matrix, read_golden
from gemm_epilogue_gb300 import inputs as gen

F16, BF16, F32 = 1, 2, 3


def enc(oracle, x, t):
    return oracle.encode(np.asarray(x, dtype=np.float64), t)


def bits_of(x, t):
    """Library conversion of exactly representable / float32 values (for pins)."""
    x = np.asarray(x, dtype=np.float64)
    if t == F16:
        return x.astype(np.float16).view(np.uint16)
    if t == BF16:
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return x.astype(np.float32)


# ---------------------------------------------------------------- formats --

def test_decode_f16_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode(pats, F16)
    want = pats.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.decode(pats, BF16)
    want = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_encode_f16_matches_numpy_direct_rounding(oracle_mod):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, 20000)),
        # exact midpoints between neighbouring half values (ties)
        (np.arange(-2048, 2048, dtype=np.float64) + 0.5) * 2.0 ** -10,
        (np.arange(0, 64, dtype=np.float64) + 0.5) * 2.0 ** -24,      # subnormal ties
        [65504.0, 65519.0, 65520.0, 65536.0, 1e9, -1e9, 2.0 ** -25, 3 * 2.0 ** -25, 0.0, -0.0],
    ])
    got = enc(oracle_mod, x, F16)
    with np.errstate(over="ignore"):  # 65520, 65536, 1e9 overflow to inf on purpose
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_bf16_matches_torch_on_float32_values(oracle_mod):
    rng = np.random.default_rng(8)
    with np.errstate(over="ignore"):  # the largest scales overflow float32; those are dropped
        x = (rng.standard_normal(20000) * np.exp2(rng.integers(-140, 128, 20000))).astype(np.float32)
    x = x[np.isfinite(x)].astype(np.float64)
    got = enc(oracle_mod, x, BF16)
    assert np.array_equal(got, bits_of(x, BF16))


def test_encode_bf16_hand_cases(oracle_mod):
    # Bit patterns worked out from the bfloat16 definition (8-bit significand).
    cases = {
        1.0 + 2.0 ** -8: 0x3F80,                 # tie -> even (1.0)
        1.0 + 3 * 2.0 ** -8: 0x3F82,             # tie -> even (1 + 2^-6)
        1.0 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,    # just above the tie: no double rounding
        -(1.0 + 2.0 ** -8 + 2.0 ** -40): 0xBF81,
        (2.0 - 2.0 ** -8) * 2.0 ** 127: 0x7F80,  # tie between max finite (odd) and 2^128 -> inf
        (2.0 - 2.0 ** -7) * 2.0 ** 127: 0x7F7F,  # max finite
        2.0 ** -134: 0x0000,                     # half the smallest subnormal: tie -> 0
        1.5 * 2.0 ** -133: 0x0002,               # tie between 1 and 2 subnormal units -> 2
        2.0 ** -126: 0x0080,                     # smallest normal
    }
    got = enc(oracle_mod, list(cases), BF16)
    assert [int(g) for g in got] == list(cases.values())


def test_encode_f16_hand_cases(oracle_mod):
    cases = {
        65520.0: 0x7C00,                          # tie between 65504 (odd) and 2^16 -> inf
        65519.0: 0x7BFF,
        2.0 ** -25: 0x0000,                       # tie -> 0
        3 * 2.0 ** -25: 0x0002,                   # tie -> 2 units
        1.0 + 2.0 ** -11 + 2.0 ** -40: 0x3C01,    # just above the tie
        -2.0: 0xC000,
    }
    got = enc(oracle_mod, list(cases), F16)
    assert [int(g) for g in got] == list(cases.values())


# ------------------------------------------------------- the worked example --

def _problem(oracle_mod, A, B, bias, ab, bt):
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    return (enc(oracle_mod, A, ab), enc(oracle_mod, B, ab),
            enc(oracle_mod, np.asarray(bias, dtype=np.float64), bt))


@pytest.mark.parametrize("ab,bt,ot", [(F16, F16, F16), (BF16, BF16, BF16), (F16, F32, F16),
                                      (BF16, F32, F32), (F16, F16, F32)])
def test_worked_example(oracle_mod, ab, bt, ot):
    g = read_golden("worked_example_2x2.txt")
    A, B, bias = (parse_matrix(g[k]) for k in ("A", "B", "bias"))
    bias = bias[0]
    a, b, bb = _problem(oracle_mod, A, B, bias, ab, bt)
    zero = enc(oracle_mod, np.zeros(2), bt)
    mm = oracle_mod.linear(a, b, zero, 2, 2, 2, ab, bt, ot)
    assert np.array_equal(oracle_mod.decode(mm.out, ot), np.array(parse_matrix(g["matmul"])))
    lin = oracle_mod.linear(a, b, bb, 2, 2, 2, ab, bt, ot)
    assert np.array_equal(oracle_mod.decode(lin.out, ot), np.array(parse_matrix(g["plus_bias"])))
    r = oracle_mod.bias_relu(a, b, bb, 2, 2, 2, ab, bt, ot)
    assert np.array_equal(oracle_mod.decode(r.out, ot), np.array(parse_matrix(g["relu"])))
    assert np.array_equal(r.ref, np.array(parse_matrix(g["relu"])))


# ------------------------------------------------------------------- K = 0 --

@pytest.mark.parametrize("ab,bt,ot", [(F16, F32, F16), (BF16, BF16, BF16), (F16, F16, F32)])
def test_k_zero_gives_relu_of_bias_on_every_row(oracle_mod, ab, bt, ot):
    # "I3 ...", "Implement in stages", stage 2: K = 0 still runs the epilogue.
    M, N = 5, 7
    bias = np.array([-3.5, -0.0, 0.0, 0.25, 1.0, -1e-3, 7.0])
    bb = enc(oracle_mod, bias, bt)
    r = oracle_mod.bias_relu(None, None, bb, M, N, 0, ab, bt, ot)
    want = enc(oracle_mod, np.maximum(oracle_mod.decode(bb, bt), 0.0), ot)
    for i in range(M):
        assert np.array_equal(r.out[i], want)
    # gate with K = 0: X = bias, out = bias + bias * Y
    Y = enc(oracle_mod, np.linspace(-2, 2, M * N).reshape(M, N), ab)
    g = oracle_mod.addmm_gate(None, None, bb, Y, M, N, 0, ab, bt, ot)
    x = 0.0 + oracle_mod.decode(bb, bt)[None, :]        # zero accumulator + bias
    assert np.array_equal(g.out, enc(oracle_mod, x + x * oracle_mod.decode(Y, ab), ot))


# ---------------------------------------------------- K = 1 versus K = 3 --

def _unfused_chain_numpy(A64, B64, b64, epi):
    """The three-step chain of library calls: matmul, + bias, then the activation."""
    x = np.matmul(A64, B64) + b64[None, :]
    return np.maximum(x, 0.0) if epi == "relu" else x


@pytest.mark.parametrize("K", [1, 3])
def test_epilogue_outside_reduction_k1_k3(oracle_mod, K):
    # "Epilogue concept", "Things that break": the same shape at K = 1 and K = 3
    # against the unfused chain; agreement at both means the epilogue is outside
    # the reduction.  Integer inputs make every value exact.
    M, N = 6, 5
    p = gen.integer_problem(M, N, K, F16, F16, seed=11 + K)
    r = oracle_mod.bias_relu(p.A, p.B, p.bias, M, N, K, F16, F16, F16)
    A64, B64, b64 = (oracle_mod.decode(x, F16) for x in (p.A, p.B, p.bias))
    want = _unfused_chain_numpy(A64, B64, b64, "relu").astype(np.float16).view(np.uint16)
    assert np.array_equal(r.out, want)
    bad = oracle_mod.bias_relu(p.A, p.B, p.bias, M, N, K, F16, F16, F16,
                               mutant=oracle_mod.MUT_BIAS_IN_SUM)
    assert np.array_equal(bad.out, want) == (K == 1)


# ------------------------------------------------------------ closed forms --

def test_closed_form_identity_A(oracle_mod):
    K = N = 9
    M = K
    rng = np.random.default_rng(3)
    Bv = rng.integers(-8, 9, (K, N)).astype(np.float64) / 4
    bv = rng.integers(-8, 9, N).astype(np.float64) / 2
    A = enc(oracle_mod, np.eye(M), BF16)
    B = enc(oracle_mod, Bv, BF16)
    b = enc(oracle_mod, bv, BF16)
    r = oracle_mod.bias_relu(A, B, b, M, N, K, BF16, BF16, F32)
    assert np.array_equal(r.ref, np.maximum(Bv + bv[None, :], 0.0))


def test_closed_form_zero_B_and_all_ones(oracle_mod):
    M, N, K = 4, 6, 37
    bv = np.array([-40.0, -37.0, -36.5, 0.0, 1.0, 3.0])
    b = enc(oracle_mod, bv, F32)
    z = oracle_mod.bias_relu(enc(oracle_mod, np.ones((M, K)), F16), enc(oracle_mod, np.zeros((K, N)), F16),
                             b, M, N, K, F16, F32, F32)
    assert np.array_equal(z.ref, np.tile(np.maximum(bv, 0), (M, 1)))
    o = oracle_mod.bias_relu(enc(oracle_mod, np.ones((M, K)), F16), enc(oracle_mod, np.ones((K, N)), F16),
                             b, M, N, K, F16, F32, F32)
    assert np.array_equal(o.ref, np.tile(np.maximum(K + bv, 0), (M, 1)))


def test_closed_form_gate_Y_zero_and_minus_one(oracle_mod):
    M, N, K = 7, 5, 12
    p = gen.random_problem(M, N, K, F16, F16, seed=5, gate=True)
    lin = oracle_mod.linear(p.A, p.B, p.bias, M, N, K, F16, F16, F32)
    y0 = np.zeros((M, N), dtype=np.uint16)                     # +0.0 in fp16
    g0 = oracle_mod.addmm_gate(p.A, p.B, p.bias, y0, M, N, K, F16, F16, F32)
    assert np.array_equal(g0.ref, lin.ref)
    y1 = enc(oracle_mod, -np.ones((M, N)), F16)
    g1 = oracle_mod.addmm_gate(p.A, p.B, p.bias, y1, M, N, K, F16, F16, F32)
    assert np.all(g1.ref == 0.0)


def test_reduction_matches_numpy_matmul(oracle_mod):
    # bias = 0, no activation: the sum is a plain matmul (library routine, fp64).
    M, N, K = 33, 29, 131
    p = gen.random_problem(M, N, K, BF16, F32, seed=9)
    zero = np.zeros(N, dtype=np.float32)
    r = oracle_mod.linear(p.A, p.B, zero, M, N, K, BF16, F32, F32)
    want = np.matmul(oracle_mod.decode(p.A, BF16), oracle_mod.decode(p.B, BF16))
    assert np.all(np.abs(r.ref - want) <= 1e-13 * (r.absdot + 1e-300))
    assert np.array_equal(r.absdot, np.matmul(np.abs(oracle_mod.decode(p.A, BF16)),
                                              np.abs(oracle_mod.decode(p.B, BF16)))) or \
        np.allclose(r.absdot, np.matmul(np.abs(oracle_mod.decode(p.A, BF16)),
                                        np.abs(oracle_mod.decode(p.B, BF16))), rtol=1e-13, atol=0)


# ------------------------------------------------------------- brute force --

def _exact(Aq, Bq, bq, i, j, K, epi, Yq=None):
    s = sum((Fraction(float(Aq[i, k])) * Fraction(float(Bq[k, j])) for k in range(K)), Fraction(0))
    v = s + Fraction(float(bq[j]))
    if epi == "relu":
        return max(v, Fraction(0))
    if epi == "gate":
        return v + v * Fraction(float(Yq[i, j]))
    return v


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 2), (5, 3, 7), (7, 9, 4), (2, 11, 13), (9, 2, 1)])
def test_brute_force_exact_tiny(oracle_mod, M, N, K):
    for ab, epi in ((F16, "relu"), (BF16, "gate")):
        p = gen.random_problem(M, N, K, ab, F32, seed=M * 100 + N * 10 + K, gate=(epi == "gate"))
        A64, B64, b64 = oracle_mod.decode(p.A, ab), oracle_mod.decode(p.B, ab), oracle_mod.decode(p.bias, F32)
        Y64 = oracle_mod.decode(p.Y, ab) if p.Y is not None else None
        if epi == "relu":
            r = oracle_mod.bias_relu(p.A, p.B, p.bias, M, N, K, ab, F32, F32)
        else:
            r = oracle_mod.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, ab, F32, F32)
        for i, j in itertools.product(range(M), range(N)):
            e = _exact(A64, B64, b64, i, j, K, epi, Y64)
            bound = 4 * K * 2.0 ** -53 * (r.absdot[i, j] + abs(b64[j])) * (1 + abs(Y64[i, j]) if Y64 is not None else 1)
            assert abs(Fraction(r.ref[i, j]) - e) <= Fraction(bound) + Fraction(0), (i, j)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (4, 7, 3), (13, 5, 9), (17, 19, 23), (40, 33, 40)])
def test_brute_force_integer_bit_exact(oracle_mod, M, N, K):
    for ab, bt, ot in ((F16, F32, F16), (BF16, BF16, BF16)):
        p = gen.integer_problem(M, N, K, ab, bt, seed=K)
        r = oracle_mod.bias_relu(p.A, p.B, p.bias, M, N, K, ab, bt, ot)
        A64, B64, b64 = oracle_mod.decode(p.A, ab), oracle_mod.decode(p.B, ab), oracle_mod.decode(p.bias, bt)
        exact = np.zeros((M, N))
        for i, j in itertools.product(range(M), range(N)):
            exact[i, j] = float(_exact(A64, B64, b64, i, j, K, "relu"))
        assert np.array_equal(r.ref, exact)
        assert np.array_equal(r.out, bits_of(exact, ot) if ot != BF16 else bits_of(exact, BF16))


# --------------------------------------------------- structure of the runs --

def test_rows_subset_and_thread_count_do_not_change_results(oracle_mod):
    M, N, K = 37, 45, 66
    p = gen.random_problem(M, N, K, F16, F16, seed=21, gate=True)
    full1 = oracle_mod.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, F16, threads=1)
    full7 = oracle_mod.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, F16, threads=7)
    assert np.array_equal(full1.out, full7.out) and np.array_equal(full1.ref, full7.ref)
    rows = [36, 0, 17, 17, 5]
    sub = oracle_mod.addmm_gate(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, F16, rows=rows)
    assert np.array_equal(sub.out, full1.out[rows])


def test_bias_broadcast_direction_rectangular(oracle_mod):
    # "Pitfalls": bias[j] not bias[i]; M != N, bias strongly column dependent.
    M, N, K = 3, 8, 2
    A = enc(oracle_mod, np.zeros((M, K)), F16)
    B = enc(oracle_mod, np.zeros((K, N)), F16)
    bias = enc(oracle_mod, np.arange(N, dtype=np.float64) - 2, F32)
    r = oracle_mod.bias_relu(A, B, bias, M, N, K, F16, F32, F32)
    assert np.array_equal(r.ref, np.tile(np.maximum(np.arange(N) - 2.0, 0), (M, 1)))


# ------------------------------------------------------------- residual add --

def test_residual_zero_equals_bias_relu(oracle_mod):
    M, N, K = 9, 13, 21
    p = gen.random_problem(M, N, K, BF16, F32, seed=70)
    zero = np.zeros((M, N), dtype=np.uint16)
    r = oracle_mod.bias_residual_relu(p.A, p.B, p.bias, zero, M, N, K, BF16, F32, BF16)
    q = oracle_mod.bias_relu(p.A, p.B, p.bias, M, N, K, BF16, F32, BF16)
    assert np.array_equal(r.out, q.out) and np.array_equal(r.ref, q.ref)


def test_residual_closed_form_and_k_zero(oracle_mod):
    # B = 0 (and K = 0): out = ReLU(bias + R), the residual added before the activation
    M, N, K = 4, 6, 5
    bias = np.array([-3.0, -1.0, 0.0, 1.0, 2.5, -0.5])
    R = np.array([[1, 2, -1, 0, -3, 0.5]] * M, dtype=np.float64) * np.arange(1, M + 1)[:, None]
    bb, Rb = enc(oracle_mod, bias, F16), enc(oracle_mod, R, F16)
    A = enc(oracle_mod, np.ones((M, K)), F16)
    B = enc(oracle_mod, np.zeros((K, N)), F16)
    want = np.maximum(bias[None, :] + R, 0.0)
    assert np.array_equal(oracle_mod.bias_residual_relu(A, B, bb, Rb, M, N, K, F16, F16, F32).ref, want)
    assert np.array_equal(oracle_mod.bias_residual_relu(None, None, bb, Rb, M, N, 0, F16, F16, F32).ref, want)


@pytest.mark.parametrize("M,N,K", [(3, 5, 2), (7, 4, 9), (11, 13, 6)])
def test_residual_brute_force_and_library_chain(oracle_mod, M, N, K):
    p = gen.integer_problem(M, N, K, F16, F16, seed=M + K, gate=True)   # Y serves as R
    r = oracle_mod.bias_residual_relu(p.A, p.B, p.bias, p.Y, M, N, K, F16, F16, F16)
    A64, B64, b64, R64 = (oracle_mod.decode(x, F16) for x in (p.A, p.B, p.bias, p.Y))
    chain = np.maximum(np.matmul(A64, B64) + b64[None, :] + R64, 0.0)
    assert np.array_equal(r.ref, chain)
    assert np.array_equal(r.out, chain.astype(np.float16).view(np.uint16))
    for i, j in itertools.product(range(M), range(N)):
        e = sum((Fraction(float(A64[i, k])) * Fraction(float(B64[k, j])) for k in range(K)), Fraction(0))
        e = max(e + Fraction(float(b64[j])) + Fraction(float(R64[i, j])), Fraction(0))
        assert Fraction(r.ref[i, j]) == e


# ------------------------------------------------------- quantized fp8 output --

E4M3 = 4


def test_decode_e4m3_every_pattern(oracle_mod):
    pats = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle_mod.decode(pats, E4M3)
    want = torch.from_numpy(pats.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_encode_e4m3_matches_torch_in_range(oracle_mod):
    rng = np.random.default_rng(12)
    x = rng.uniform(-448, 448, 20000) * np.exp2(rng.integers(-14, 1, 20000))
    ties = [(m + 0.5) * 2.0 ** -9 for m in range(8)] + [(8 + m + 0.5) * 2.0 ** (e - 10)
                                                     for e in range(1, 16) for m in range(7)]
    x = np.concatenate([x, ties, -np.array(ties)]).astype(np.float32).astype(np.float64)
    x = x[np.abs(x) <= 448]
    got = oracle_mod.encode(x, E4M3)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_encode_e4m3_hand_cases(oracle_mod):
    # worked out from the e4m3 definition (4 significand bits, largest finite 448, no inf)
    cases = {464.0: 0x7E,                     # tie between 448 (even) and 480 (not finite) -> 448
             1000.0: 0x7E, -1e9: 0xFE,         # saturate (satfinite)
             2.0 ** -10: 0x00,                 # half the smallest subnormal: tie -> 0
             3 * 2.0 ** -10: 0x02,             # tie between 1 and 2 subnormal units -> 2
             0.5 + 2.0 ** -5: 0x30,            # tie between 0.5 and 0.5625 -> 0.5 (even)
             0.5 + 2.0 ** -5 + 2.0 ** -30: 0x31,
             2.0 ** -6: 0x08, 448.0: 0x7E, -2.0: 0xC0}
    got = oracle_mod.encode(np.array(list(cases)), E4M3)
    assert [int(g) for g in got] == list(cases.values())


@pytest.mark.parametrize("scale", [0.25, 1.0, 8.0])
def test_quant_epilogue_against_library_chain(oracle_mod, scale):
    # "Variants": matmul + quantized output; integer inputs and power-of-two scales are exact
    M, N, K = 9, 14, 5
    p = gen.integer_problem(M, N, K, BF16, F32, seed=int(scale * 4))
    r = oracle_mod.bias_relu_quant(p.A, p.B, p.bias, M, N, K, BF16, F32, scale)
    A64, B64, b64 = oracle_mod.decode(p.A, BF16), oracle_mod.decode(p.B, BF16), oracle_mod.decode(p.bias, F32)
    v = np.clip(scale * np.maximum(A64 @ B64 + b64[None, :], 0.0), -448, 448)
    assert np.array_equal(r.ref, v)
    assert np.array_equal(r.out, torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn)
                          .view(torch.uint8).numpy())


def test_quant_closed_forms(oracle_mod):
    M, N, K = 3, 5, 4
    bias = np.array([-1.0, 0.0, 3.0, 100.0, 1e4])
    A = enc(oracle_mod, np.zeros((M, K)), F16)
    B = enc(oracle_mod, np.ones((K, N)), F16)
    r = oracle_mod.bias_relu_quant(A, B, enc(oracle_mod, bias, F32), M, N, K, F16, F32, 2.0)
    assert np.array_equal(r.ref, np.tile([0.0, 0.0, 6.0, 200.0, 448.0], (M, 1)))   # clamp at 448
    assert np.array_equal(oracle_mod.decode(r.out, E4M3), np.tile([0.0, 0.0, 6.0, 192.0, 448.0], (M, 1)))



# ------------------------------------------------------------- fp8 operands --

@pytest.mark.parametrize("K", [1, 17, 64])
def test_e4m3_operands_against_library_decode(oracle_mod, K):
    # fp8 operands ("Optimizing GEMM + Activation on CDNA4 with TLX", "Future Work": half the
    # operand bytes): every finite e4m3 pattern is drawn, decoded by torch's own float8 type, and
    # the fp64 matmul of the decoded values is exact here (a product of two e4m3 values has at most
    # 8 significant bits between 2^-18 and 2^17, and 64 of them sum exactly in 53 bits).
    M, N = 7, 12
    rng = np.random.default_rng(300 + K)
    finite = np.array([p for p in range(256) if p & 0x7F != 0x7F], dtype=np.uint8)
    A = rng.choice(finite, (M, K))
    B = rng.choice(finite, (K, N))
    bias = rng.standard_normal(N).astype(np.float32)
    r = oracle_mod.bias_relu(A, B, bias, M, N, K, E4M3, F32, F32)
    dec = lambda x: torch.from_numpy(x.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    want = np.maximum(dec(A) @ dec(B) + bias.astype(np.float64)[None, :], 0.0)
    assert np.array_equal(r.ref, want)
    # and the one rounding to fp32 is round-to-nearest of that exact value
    assert np.array_equal(r.out, want.astype(np.float32))


def test_e4m3_operands_transposed_b_is_caught(oracle_mod):
    # a square B and its transpose give different products: the oracle must read B as K x N
    M = N = K = 6
    rng = np.random.default_rng(310)
    finite = np.array([p for p in range(256) if p & 0x7F != 0x7F], dtype=np.uint8)
    A, B = rng.choice(finite, (M, K)), rng.choice(finite, (K, N))
    bias = np.zeros(N, dtype=np.float32)
    dec = lambda x: torch.from_numpy(x.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    r = oracle_mod.gemm_epilogue(A, B, bias, M, N, K, E4M3, F32, F32, oracle_mod.EPI_LINEAR)
    assert np.array_equal(r.ref, dec(A) @ dec(B))
    assert not np.array_equal(r.ref, dec(A) @ dec(B).T)


@pytest.mark.parametrize("K", [1, 13, 64])
@pytest.mark.parametrize("yt", [F16, BF16])
def test_e4m3_gate_with_16_bit_y(oracle_mod, K, yt):
    # "Optimizing GEMM + Activation on CDNA4 with TLX", "Future Work" (FP8 precision): the
    # projection A @ B in fp8 while the gate's Y stays 16-bit.  Y is decoded by its own type: the
    # result equals torch's float8 decode of A and B, an fp64 matmul (exact here), the bias, and
    # X + X * Y with Y decoded by numpy / torch; reading Y as the other 16-bit type must differ.
    M, N = 6, 10
    rng = np.random.default_rng(500 + K + yt)
    finite = np.array([p for p in range(256) if p & 0x7F != 0x7F], dtype=np.uint8)
    A, B = rng.choice(finite, (M, K)), rng.choice(finite, (K, N))
    bias = rng.standard_normal(N).astype(np.float32)
    Yf = rng.standard_normal((M, N)).astype(np.float32)
    if yt == F16:
        Y = Yf.astype(np.float16).view(np.uint16)
        Y64 = Y.view(np.float16).astype(np.float64)
    else:
        Y = torch.from_numpy(Yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
        Y64 = torch.from_numpy(Y.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    r = oracle_mod.addmm_gate(A, B, bias, Y, M, N, K, E4M3, F32, F32, y_type=yt)
    dec = lambda x: torch.from_numpy(x.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    X = dec(A) @ dec(B) + bias.astype(np.float64)[None, :]
    assert np.array_equal(r.ref, X + X * Y64)
    other = oracle_mod.addmm_gate(A, B, bias, Y, M, N, K, E4M3, F32, F32,
                                  y_type=BF16 if yt == F16 else F16)
    assert not np.array_equal(other.ref, r.ref)
    # residual with a 16-bit R beside fp8 operands
    rr = oracle_mod.bias_residual_relu(A, B, bias, Y, M, N, K, E4M3, F32, F32, y_type=yt)
    assert np.array_equal(rr.ref, np.maximum(X + Y64, 0.0))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 2), (5, 3, 7), (4, 9, 16)])
def test_e4m3_gate_brute_force_exact(oracle_mod, M, N, K):
    # exact rational arithmetic on the decoded values (fp8 operands, 16-bit Y, fp32 bias)
    rng = np.random.default_rng(600 + M * N * K)
    finite = np.array([p for p in range(256) if p & 0x7F != 0x7F], dtype=np.uint8)
    A, B = rng.choice(finite, (M, K)), rng.choice(finite, (K, N))
    bias = rng.standard_normal(N).astype(np.float32)
    Y = rng.standard_normal((M, N)).astype(np.float16).view(np.uint16)
    r = oracle_mod.addmm_gate(A, B, bias, Y, M, N, K, E4M3, F32, F32, y_type=F16)
    A64, B64 = oracle_mod.decode(A, E4M3), oracle_mod.decode(B, E4M3)
    b64, Y64 = oracle_mod.decode(bias, F32), oracle_mod.decode(Y, F16)
    for i, j in itertools.product(range(M), range(N)):
        e = _exact(A64, B64, b64, i, j, K, "gate", Y64)
        x = _exact(A64, B64, b64, i, j, K, "linear")
        # three fp64 roundings at most (the bias add, X * Y, the final add; the products and
        # their sum are exact): bounded by the magnitudes they act on
        bound = 4 * 2.0 ** -53 * abs(float(x)) * (1 + abs(Y64[i, j])) + 1e-300
        assert abs(Fraction(r.ref[i, j]) - e) <= Fraction(bound), (i, j)


# --------------------------------------------------------- negative controls --

def _pins_pass(oracle_mod, mutant):
    """Run a compact set of the pins above against the (possibly mutated) oracle."""
    ok = True
    # worked example
    g = read_golden("worked_example_2x2.txt")
    a, b, bb = _problem(oracle_mod, parse_matrix(g["A"]), parse_matrix(g["B"]),
                        parse_matrix(g["bias"])[0], F16, F16)
    r = oracle_mod.bias_relu(a, b, bb, 2, 2, 2, F16, F16, F32, mutant=mutant)
    ok &= np.array_equal(r.ref, np.array(parse_matrix(g["relu"])))
    # K = 0 and K = 3 against the unfused chain (integer inputs)
    for K in (0, 1, 3):
        p = gen.integer_problem(6, 5, K, F16, F16, seed=40 + K)
        rr = oracle_mod.bias_relu(p.A, p.B, p.bias, 6, 5, K, F16, F16, F32, mutant=mutant)
        A64 = oracle_mod.decode(p.A, F16)
        B64 = oracle_mod.decode(p.B, F16)
        want = _unfused_chain_numpy(A64, B64, oracle_mod.decode(p.bias, F16), "relu")
        ok &= np.array_equal(rr.ref, want)
    # gate closed forms and brute force
    p = gen.integer_problem(5, 4, 3, F16, F16, seed=50, gate=True)
    gg = oracle_mod.addmm_gate(p.A, p.B, p.bias, p.Y, 5, 4, 3, F16, F16, F32, mutant=mutant)
    A64, B64, b64, Y64 = (oracle_mod.decode(x, F16) for x in (p.A, p.B, p.bias, p.Y))
    X = A64 @ B64 + b64[None, :]
    ok &= np.array_equal(gg.ref, X + X * Y64)
    # residual: added before the activation, checked against the library chain
    p = gen.integer_problem(5, 4, 3, F16, F16, seed=51, gate=True)
    rr = oracle_mod.bias_residual_relu(p.A, p.B, p.bias, p.Y, 5, 4, 3, F16, F16, F32, mutant=mutant)
    A64, B64, b64, R64 = (oracle_mod.decode(x, F16) for x in (p.A, p.B, p.bias, p.Y))
    ok &= np.array_equal(rr.ref, np.maximum(A64 @ B64 + b64[None, :] + R64, 0.0))
    # quantized output: scale after bias and activation
    p = gen.integer_problem(6, 5, 3, BF16, F32, seed=52)
    qq = oracle_mod.bias_relu_quant(p.A, p.B, p.bias, 6, 5, 3, BF16, F32, 0.5, mutant=mutant)
    A64, B64, b64 = oracle_mod.decode(p.A, BF16), oracle_mod.decode(p.B, BF16), oracle_mod.decode(p.bias, F32)
    ok &= np.array_equal(qq.ref, np.clip(0.5 * np.maximum(A64 @ B64 + b64[None, :], 0), -448, 448))
    # rectangular non-symmetric matmul against numpy (catches transposed operands)
    p = gen.random_problem(7, 5, 9, BF16, F32, seed=60)
    zero = np.zeros(5, dtype=np.float32)
    ll = oracle_mod.linear(p.A, p.B, zero, 7, 5, 9, BF16, F32, F32, mutant=mutant)
    want = oracle_mod.decode(p.A, BF16) @ oracle_mod.decode(p.B, BF16)
    ok &= bool(np.allclose(ll.ref, want, rtol=1e-12, atol=1e-12))
    return bool(ok)


def test_pins_accept_the_oracle(oracle_mod):
    assert _pins_pass(oracle_mod, oracle_mod.OK)


@pytest.mark.parametrize("name", ["relu_first", "bias_row", "bias_in_sum", "drop_gemm",
                                  "transpose_b", "drop_last_k", "gate_sign", "resid_after",
                                  "scale_first"])
def test_pins_reject_each_planted_mistake(oracle_mod, name):
    assert not _pins_pass(oracle_mod, oracle_mod.MUTANTS[name])
