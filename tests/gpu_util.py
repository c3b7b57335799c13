"""Helpers for the GPU parity tests: uploads, tolerance checks against the oracle."""
import math

import numpy as np

import oracle

F16, BF16, F32, E4M3 = 1, 2, 3, 4


def torch_dtype(t):
    import torch
    return {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32, E4M3: torch.uint8}[t]


def up(a, t, dev="cuda"):
    """numpy bits (uint16) or float32 -> device tensor of type t."""
    import torch
    if a is None:
        return None
    if t == F32:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    if t == E4M3:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch_dtype(t)).to(dev)


def down(x, t):
    """device tensor -> numpy bits (uint16) or float32."""
    import torch
    x = x.detach().cpu().contiguous()
    if t == F32:
        return x.numpy().astype(np.float32)
    if t == E4M3:
        return x.numpy().astype(np.uint8)
    return x.view(torch.int16).numpy().view(np.uint16)


def dtype_word(ab, bias, out, y=None):
    """The library's dtype word; `y` is the gate's Y type when it is not the operand type."""
    import gemm_epilogue_gb300.binding as fg
    w = {F16: fg.F16, BF16: fg.BF16, E4M3: fg.E4M3}[ab]
    if y is not None and y != ab:
        w |= {F16: fg.Y_F16, BF16: fg.Y_BF16}[y]
    if bias == F32:
        w |= fg.BIAS_F32
    elif bias == BF16 and ab != BF16:
        w |= fg.BIAS_BF16
    elif bias != ab:
        raise ValueError("unsupported bias type")
    if out == F32:
        w |= fg.OUT_F32
    elif out == E4M3:
        w |= fg.OUT_E4M3
    elif out == BF16 and ab != BF16:
        w |= fg.OUT_BF16
    elif out == F16 and ab != F16:
        w |= fg.OUT_F16
    elif out != ab:
        raise ValueError("unsupported out type")
    return w


def ulp(x, t):
    """Spacing of type t at |x| (the gap to the next representable magnitude)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    p, emin = {F16: (11, -14), BF16: (8, -126), F32: (24, -126), E4M3: (4, -6)}[t]
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** emin)))
    return np.exp2(np.maximum(e, emin) - (p - 1))


def tolerance(K, ref_vals, out_type):
    """Stated tolerance: max|err| <= 2e-2 sqrt(K/4096) max|ref| + 1e-3 (16-bit outputs),
    1e-4 relative for fp32 outputs."""
    m = float(np.abs(ref_vals).max()) if ref_vals.size else 0.0
    if out_type == F32:
        return 1e-4 * m
    return 2e-2 * math.sqrt(K / 4096.0) * m + 1e-3


def check_close(got_bits, res, K, out_type, Y64=None, bias64=None, what=""):
    """Stated tolerance plus the per-element forward-error bound.

    Secondary bound per element: |gpu - oracle| <= 1 ulp(out) + K * 2^-22 * (sum|a b| + |bias|)
    * (1 + |y|): an fp32 recursive sum of K products (with a margin for the tensor core's
    accumulation) and one rounding of each result to the output type.
    """
    got = oracle.decode(got_bits, out_type)
    ref = oracle.decode(res.out, out_type)
    err = np.abs(got - ref)
    tol = tolerance(K, ref, out_type)
    worst = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert worst <= tol, f"{what}: max|err| {worst:.4g} > tolerance {tol:.4g}"
    scale = res.absdot + (np.abs(bias64)[None, :] if bias64 is not None else 0.0)
    if Y64 is not None:
        scale = scale * (1.0 + np.abs(Y64))
    bound = ulp(np.maximum(np.abs(ref), np.abs(got)), out_type) + K * 2.0 ** -22 * scale + 1e-30
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements exceed the forward-error bound " \
                          f"(first at {np.argwhere(bad)[0]}, err {err[bad][0]:.3g}, bound {bound[bad][0]:.3g})"
    return worst, tol


def sample_rows(M, BM=128, n_random=64, seed=0):
    """Rows for full-size parity, stratified over the tile grid: in every BM-row M tile one
    seeded row from each 32-row quarter (each quarter is read out of tensor memory by its own
    epilogue warp, so every warp of every M tile is sampled), every row of the last (ragged)
    M tile, the first and last rows, and `n_random` more seeded rows anywhere."""
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    for t0 in range(0, M, BM):
        for q0 in range(t0, min(t0 + BM, M), 32):
            rows.add(int(rng.integers(q0, min(q0 + 32, M))))
    rows.update(range(max(0, (M - 1) // BM * BM), M))
    rows.update(int(r) for r in rng.integers(0, M, min(n_random, M)))
    return np.array(sorted(rows), dtype=np.int64)


NAN_BITS = {F16: 0x7FFF, BF16: 0x7FFF, F32: 0x7FFFFFFF, E4M3: 0x7F}
GUARD = 4096


def guarded_out(M, N, t, dev="cuda"):
    """An M x N output tensor of type t inside a buffer of raw words pre-filled with a NaN bit
    pattern, with GUARD elements of that pattern on both sides.  Returns (out, buf)."""
    import torch
    word = {F16: torch.int16, BF16: torch.int16, F32: torch.int32, E4M3: torch.uint8}[t]
    buf = torch.full((GUARD + M * N + GUARD,), NAN_BITS[t], dtype=word, device=dev)
    inner = buf[GUARD:GUARD + M * N]
    out = inner if t == E4M3 else inner.view(torch_dtype(t))
    return out.view(M, N), buf


def check_guarded(buf, M, N, t, what=""):
    """Every element of out written (no NaN pattern left: the outputs here are finite) and
    nothing written outside it (the guard words keep their bits)."""
    import torch
    b = buf.cpu()
    for g in (b[:GUARD], b[GUARD + M * N:]):
        assert bool((g == NAN_BITS[t]).all()), f"{what}: a guard element was written"
    inner = b[GUARD:GUARD + M * N]
    if t == E4M3:
        nan = (inner & 0x7F) == 0x7F
    else:
        nan = torch.isnan(inner.view(torch_dtype(t)))
    assert not bool(nan.any()), f"{what}: {int(nan.sum())} output elements never written"
