"""Pins for the CPU oracle: each check compares it with something other than
itself -- IEEE encodings, exact rational brute force, closed forms, layout
invariance, hand-worked traces from the pages' formulas, and torch's own
rounding for cases where no double rounding is possible."""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

K, MN = oracle.K_CONTIG, oracle.MN_CONTIG


# ---------------------------------------------------------------- decoding

def test_decode_ieee_bit_patterns():
    f16 = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF, 0x3555], dtype=np.uint16)
    got = oracle.decode(f16, oracle.F16)
    assert got.tolist() == [1.0, -2.0, 2.0 ** -24, 65504.0, struct.unpack("<e", struct.pack("<H", 0x3555))[0]]
    bf = np.array([0x3F80, 0xC040, 0x4049, 0x0001, 0x7F7F], dtype=np.uint16)
    got = oracle.decode(bf, oracle.BF16)
    assert got[0] == 1.0 and got[1] == -3.0
    assert got[2] == 3.140625
    assert got[3] == 2.0 ** -133
    assert got[4] == (2 - 2 ** -7) * 2.0 ** 127


def test_decode_torch_tensors():
    x = torch.tensor([1.5, -0.25, 3.0], dtype=torch.bfloat16)
    assert oracle.decode(x, oracle.BF16).tolist() == [1.5, -0.25, 3.0]
    y = torch.tensor([1.5, -0.25, 3.0], dtype=torch.float16)
    assert oracle.decode(y, oracle.F16).tolist() == [1.5, -0.25, 3.0]


def test_round_to_bf16_matches_torch_on_binary32_inputs():
    # Inputs exactly representable in binary32: torch's single rounding
    # binary32 -> bf16 is then the same problem.
    g = torch.Generator().manual_seed(5)
    x32 = torch.randn(200000, generator=g, dtype=torch.float32) * torch.exp2(
        torch.randint(-40, 40, (200000,), generator=g).float())
    ties = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 1.5], dtype=torch.float32)
    x32 = torch.cat([x32, ties])
    want = x32.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to(x32.double().numpy(), oracle.BF16)
    assert np.array_equal(got, want)


def test_round_to_bf16_single_rounding_from_fp64():
    # 1 + 2^-8 + 2^-40 is above the tie: one rounding goes up; a detour via
    # binary32 would round to the tie and then to even (down).
    x = np.array([1 + 2 ** -8 + 2 ** -40])
    assert oracle.round_to(x, oracle.BF16)[0] == 1 + 2 ** -7


def test_round_to_f16_ties_even():
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 2049.0, 2051.0, 70000.0])
    got = oracle.round_to(x, oracle.F16)
    assert got[:4].tolist() == [1.0, 1 + 2 ** -9, 2048.0, 2052.0]
    assert np.isinf(got[4])


# ---------------------------------------------------------------- GEMM pins

def _store(logical: np.ndarray, layout_k_rows: bool, ld: int, dtype):
    """Place a logical R x C matrix (values already in dtype) into a flat
    storage buffer, independently of the oracle's index functions: build the
    storage matrix with numpy and copy it into a padded row buffer."""
    mat = logical if layout_k_rows else logical.T
    rows, cols = mat.shape
    buf = np.full((rows, ld), np.nan, dtype=np.float64)
    buf[:, :cols] = mat
    t = torch.from_numpy(buf.reshape(-1)).to(wl.TORCH_DTYPE[dtype])
    return t


def _store_a(a, layout, ld, dtype):
    # K-contig: rows are m (M x K as is); M-contig: rows are k (K x M)
    return _store(a, layout == K, ld, dtype)


def _store_b(b, layout, ld, dtype):
    # b is logical K x N.  K-contig: rows are n (N x K); N-contig: rows are k.
    return _store(b.T, True, ld, dtype) if layout == K else _store(b, True, ld, dtype)


def _f16_exact(bits):
    return Fraction(struct.unpack("<e", struct.pack("<H", int(bits)))[0])


def _bf16_exact(bits):
    return Fraction(struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0])


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
@pytest.mark.parametrize("a_layout", [K, MN])
@pytest.mark.parametrize("b_layout", [K, MN])
def test_gemm_bruteforce_exact_tiny(dtype, a_layout, b_layout):
    """Exact rational dot products, decoding each stored element with the
    struct module, on every shape up to 4 x 4 x 5 with padded leading dims."""
    rng = np.random.default_rng(1 + 4 * dtype + 2 * a_layout + b_layout)
    exact = _f16_exact if dtype == oracle.F16 else _bf16_exact
    for M in (1, 2, 4):
        for N in (1, 3, 4):
            for Kd in (1, 2, 5):
                a = rng.uniform(-1, 1, (M, Kd))
                b = rng.uniform(-1, 1, (Kd, N))
                lda = (Kd if a_layout == K else M) + 3
                ldb = (Kd if b_layout == K else N) + 2
                A = _store_a(a, a_layout, lda, dtype)
                B = _store_b(b, b_layout, ldb, dtype)
                got = oracle.gemm(M, N, Kd, A, a_layout, lda, dtype, B, b_layout, ldb, dtype)
                Ab = A.view(torch.int16).numpy().view(np.uint16)
                Bb = B.view(torch.int16).numpy().view(np.uint16)
                for m in range(M):
                    for n in range(N):
                        s = Fraction(0)
                        for k in range(Kd):
                            ai = m * lda + k if a_layout == K else k * lda + m
                            bi = n * ldb + k if b_layout == K else k * ldb + n
                            s += exact(Ab[ai]) * exact(Bb[bi])
                        assert abs(Fraction(got[m, n]) - s) <= abs(s) * Fraction(1, 2 ** 50)


def test_gemm_identity_and_permutation_closed_forms():
    rng = np.random.default_rng(7)
    n = 24
    b = rng.uniform(-1, 1, (n, 17))
    ident = np.eye(n)
    for al in (K, MN):
        for bl in (K, MN):
            lda = n + (1 if al == K else 5)
            ldb = (n if bl == K else 17) + 4
            A = _store_a(ident, al, lda, oracle.F16)
            B = _store_b(b, bl, ldb, oracle.F16)
            C = oracle.gemm(n, 17, n, A, al, lda, oracle.F16, B, bl, ldb, oracle.F16)
            assert np.array_equal(C, oracle.round_to(b, oracle.F16))      # I.B = B
    # B = permutation matrix: C's columns are A's columns permuted
    sigma = rng.permutation(n)
    P = np.zeros((n, n))
    P[sigma, np.arange(n)] = 1.0          # column j of P selects row sigma[j]
    a = rng.uniform(-1, 1, (9, n))
    for al in (K, MN):
        for bl in (K, MN):
            lda = (n if al == K else 9)
            ldb = n
            C = oracle.gemm(9, n, n, _store_a(a, al, lda, oracle.BF16), al, lda, oracle.BF16,
                            _store_b(P, bl, ldb, oracle.BF16), bl, ldb, oracle.BF16)
            assert np.array_equal(C, oracle.round_to(a, oracle.BF16)[:, sigma])


def test_gemm_all_ones_gives_K_and_unit_selector():
    for Kd in (1, 7, 256, 3000):
        ones_a = np.ones((5, Kd))
        ones_b = np.ones((Kd, 3))
        C = oracle.gemm(5, 3, Kd, _store_a(ones_a, MN, 5, oracle.F16), MN, 5, oracle.F16,
                        _store_b(ones_b, K, Kd, oracle.F16), K, Kd, oracle.F16)
        assert np.all(C == Kd)
    # A = e_i e_j^T picks row j of B into row i of C
    rng = np.random.default_rng(3)
    b = rng.uniform(-2, 2, (6, 5))
    a = np.zeros((4, 6))
    a[2, 4] = 1.0
    C = oracle.gemm(4, 5, 6, _store_a(a, K, 6, oracle.F16), K, 6, oracle.F16,
                    _store_b(b, MN, 5, oracle.F16), MN, 5, oracle.F16)
    want = np.zeros((4, 5))
    want[2] = oracle.round_to(b[4], oracle.F16)
    assert np.array_equal(C, want)


def test_gemm_layout_invariance():
    """The same logical A and B stored in all four layouts (and with padded
    leading dimensions) give bit-identical results."""
    rng = np.random.default_rng(11)
    M, N, Kd = 37, 29, 53
    a = rng.normal(size=(M, Kd))
    b = rng.normal(size=(Kd, N))
    outs = []
    for al in (K, MN):
        for bl in (K, MN):
            for pad in (0, 3):
                lda = (Kd if al == K else M) + pad
                ldb = (Kd if bl == K else N) + pad
                outs.append(oracle.gemm(M, N, Kd, _store_a(a, al, lda, oracle.BF16), al, lda, oracle.BF16,
                                        _store_b(b, bl, ldb, oracle.BF16), bl, ldb, oracle.BF16))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_planted_layout_mistake_is_caught(monkeypatch):
    """Swap the two A addressing formulas in the oracle: the brute-force and
    invariance pins must then fail."""
    real = oracle.a_index

    def swapped(m, k, layout, lda):
        return real(m, k, 1 - layout, lda)

    monkeypatch.setattr(oracle, "a_index", swapped)
    rng = np.random.default_rng(2)
    a = rng.normal(size=(5, 5))
    b = rng.normal(size=(5, 3))
    A = _store_a(a, K, 5, oracle.F16)
    C = oracle.gemm(5, 3, 5, A, K, 5, oracle.F16, _store_b(b, K, 5, oracle.F16), K, 5, oracle.F16)
    want = oracle.round_to(a, oracle.F16) @ oracle.round_to(b, oracle.F16)
    assert not np.allclose(C, want)


def test_planted_dequant_mistake_is_caught(monkeypatch):
    """Drop the zero point from the dequantisation: the all-8 codes pin fails."""
    def no_zero(W, scales, zeros, N, K_, group):
        q = oracle.int4_codes(W, N, K_).astype(np.float64)
        s = oracle.decode(scales, oracle.F16).reshape(N, K_ // group)
        return (q * s[:, np.arange(K_) // group]).T

    monkeypatch.setattr(oracle, "dequant_int4", no_zero)
    A = _store_a(np.ones((1, 128)), K, 128, oracle.F16)
    W8 = np.full(4 * 64, 0x88, dtype=np.uint8)
    s = torch.full((4, 1), 0.01, dtype=torch.float16)
    C = oracle.gemm(1, 4, 128, A, K, 128, oracle.F16, W8, K, 0, oracle.INT4, scales=s)
    assert not np.all(C == 0)


def test_gemm_elements_matches_full():
    case = wl.GemmCase("t", 70, 45, 130, MN, K, oracle.BF16, oracle.BF16, oracle.BF16,
                       ("normal", 1.0), ("normal", 1.0), lda=75, ldb=131)
    inp = wl.make_inputs(case, seed=2)
    full = oracle.gemm(70, 45, 130, inp.A, MN, inp.lda, oracle.BF16, inp.B, K, inp.ldb, oracle.BF16)
    rows, cols = wl.sample_indices(70, 45, 50)
    el = oracle.gemm_elements(rows, cols, 70, 45, 130, inp.A, MN, inp.lda, oracle.BF16, inp.B, K, inp.ldb,
                              oracle.BF16)
    assert np.allclose(el, full[rows, cols], rtol=1e-13, atol=1e-13)
    assert np.all(np.isfinite(full))       # NaN padding was never read


def test_gemm_k_zero_is_zero():
    C = oracle.gemm(3, 4, 0, torch.zeros(0, dtype=torch.float16), K, 1, oracle.F16,
                    torch.zeros(0, dtype=torch.float16), K, 1, oracle.F16)
    assert C.shape == (3, 4) and np.all(C == 0)


# ---------------------------------------------------------------- int4

def test_int4_nibble_order_and_codes():
    # byte 0x21: k=0 -> 1 (low nibble), k=1 -> 2; byte 0xF0: k=2 -> 0, k=3 -> 15
    W = np.array([0x21, 0xF0, 0x88, 0x7E], dtype=np.uint8)
    q = oracle.int4_codes(W, 1, 8)
    assert q.tolist() == [[1, 2, 0, 15, 8, 8, 14, 7]]


def test_int4_zero_codes_give_zero_and_constant_codes_give_scaled_sum():
    N, Kd, g = 8, 256, 128
    rng = np.random.default_rng(4)
    a = rng.uniform(-1, 1, (3, Kd))
    A = _store_a(a, K, Kd, oracle.F16)
    W8 = np.full(N * Kd // 2, 0x88, dtype=np.uint8)
    s = torch.full((N, Kd // g), 0.01, dtype=torch.float16)
    C = oracle.gemm(3, N, Kd, A, K, Kd, oracle.F16, W8, K, 0, oracle.INT4, scales=s, zeros=None, group=g)
    assert np.all(C == 0)
    W9 = np.full(N * Kd // 2, 0x99, dtype=np.uint8)
    s64 = torch.full((N, Kd // g), 1.0 / 64, dtype=torch.float16)
    z = torch.full((N, Kd // g), 8.0, dtype=torch.float16)
    C = oracle.gemm(3, N, Kd, A, K, Kd, oracle.F16, W9, K, 0, oracle.INT4, scales=s64, zeros=z, group=g)
    want = oracle.round_to(a, oracle.F16).sum(axis=1) / 64
    assert np.allclose(C, want[:, None], rtol=0, atol=1e-14)


def test_int4_group_indexing():
    """Only group 1 of row n=2 is non-zero: C[:, 2] equals the dot product of
    A's k in [128, 256) with (q - z) * s, every other column is zero."""
    N, Kd, g = 4, 384, 128
    rng = np.random.default_rng(8)
    a = rng.uniform(-1, 1, (2, Kd))
    A = _store_a(a, K, Kd, oracle.F16)
    W = np.full((N, Kd // 2), 0x88, dtype=np.uint8)
    codes = rng.integers(0, 16, size=g)
    W[2, 64:128] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    s = torch.full((N, 3), 0.5, dtype=torch.float16)
    s[2, 1] = 0.125
    z = torch.full((N, 3), 8.0, dtype=torch.float16)
    z[2, 1] = 3.0
    C = oracle.gemm(2, N, Kd, A, K, Kd, oracle.F16, W.reshape(-1), K, 0, oracle.INT4, scales=s, zeros=z, group=g)
    af = oracle.round_to(a, oracle.F16)
    want2 = af[:, 128:256] @ ((codes - 3.0) * 0.125)
    assert np.allclose(C[:, 2], want2, rtol=1e-14, atol=1e-14)
    assert np.all(C[:, [0, 1, 3]] == 0)


def test_int4_elements_match_full():
    case = wl.GemmCase("t4", 5, 40, 256, K, K, oracle.F16, oracle.INT4, oracle.F16, ("normal", 1.0), ("bytes",))
    inp = wl.make_inputs(case, 3)
    full = oracle.gemm(5, 40, 256, inp.A, K, inp.lda, oracle.F16, inp.B, K, 0, oracle.INT4,
                       scales=inp.scales, zeros=inp.zeros)
    rows, cols = wl.sample_indices(5, 40, 30)
    el = oracle.gemm_elements(rows, cols, 5, 40, 256, inp.A, K, inp.lda, oracle.F16, inp.B, K, 0, oracle.INT4,
                              scales=inp.scales, zeros=inp.zeros)
    assert np.allclose(el, full[rows, cols], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- split-K rule

def _read_traces(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "splitk_traces.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            head, result = line.split("->")
            parts = head.split()
            M, N, Kd, sms = map(int, parts[:4])
            trace = []
            for item in parts[4:]:
                fac, frac = item.split(":")
                w, t = frac.split("/")
                trace.append((int(fac), int(w), int(t)))
            out.append((M, N, Kd, sms, trace, int(result)))
    return out


def test_splitk_hand_traces(golden_dir):
    cases = _read_traces(golden_dir)
    assert len(cases) >= 10
    for M, N, Kd, sms, trace, want in cases:
        assert oracle.splitk_factor(M, N, Kd, 128, 128, 64, sms, 0.05) == want, (M, N, Kd, sms)
        got = oracle.splitk_trace(M, N, Kd, 128, 128, 64, sms, 0.05)
        assert [f for f, _ in got] == [f for f, _, _ in trace]
        for (f, r), (_, w, t) in zip(got, trace):
            assert r == w / t


def test_splitk_properties():
    rng = np.random.default_rng(0)
    for _ in range(3000):
        M, N = int(rng.integers(1, 9000)), int(rng.integers(1, 9000))
        Kd = int(rng.integers(1, 70000))
        sms = int(rng.integers(1, 200))
        f = oracle.splitk_factor(M, N, Kd, 128, 128, 64, sms)
        assert f >= 1 and (f & (f - 1)) == 0
        t = -(-M // 128) * -(-N // 128) * f
        assert (t % sms) / t <= 0.05 or 2 * f * 64 >= Kd
        if f > 1:       # the previous factor failed the ratio and passed the K test
            tp = t // 2
            assert (tp % sms) / tp > 0.05 and f * 64 < Kd


# ---------------------------------------------------------------- permutation

def _read_perm(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "perm_examples.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            head, vals = line.split(":")
            B, S = map(int, head.split())
            out.append((B, S, [int(v) for v in vals.split()]))
    return out


def test_perm_worked_examples(golden_dir):
    ex = _read_perm(golden_dir)
    assert len(ex) >= 5
    for B, S, want in ex:
        assert [oracle.perm_forward(i, B, S) for i in range(B)] == want
        assert [oracle.perm_inverse(want[i], B, S) for i in range(B)] == list(range(B))


def test_perm_is_grid_transpose_exhaustive():
    """Forward map = transpose of a (B/S) x S index grid, for every B <= 256
    and every S dividing B; inverse undoes it; both are bijections."""
    for B in range(1, 257):
        for S in range(1, B + 1):
            if B % S:
                continue
            fwd = [oracle.perm_forward(i, B, S) for i in range(B)]
            closed = np.arange(B).reshape(B // S, S).T.ravel().tolist()
            assert fwd == closed
            assert sorted(fwd) == list(range(B))
            assert [oracle.perm_inverse(v, B, S) for v in fwd] == list(range(B))


def test_perm_blocks_and_tail():
    got = oracle.perm_apply(20, 8, 2)
    assert got[:8] == [0, 2, 4, 6, 1, 3, 5, 7]
    assert got[8:16] == [8 + v for v in [0, 2, 4, 6, 1, 3, 5, 7]]
    assert got[16:] == [16, 17, 18, 19]
    with pytest.raises(ValueError):
        oracle.perm_forward(0, 8, 3)


# ---------------------------------------------------------------- acceptance

def test_check_close_catches_planted_errors():
    rng = np.random.default_rng(1)
    ref = rng.normal(size=(64, 64)) * 30
    ok, _, _ = oracle.check_close(oracle.round_to(ref, oracle.BF16), ref)
    assert ok
    bad = oracle.round_to(ref, oracle.BF16)
    bad[3, 4] += 0.05 * (abs(ref[3, 4]) + 1)
    assert not oracle.check_close(bad, ref)[0]
    bad2 = ref * (1 + 3e-3)
    assert not oracle.check_close(bad2, ref)[0]
    nan = ref.copy()
    nan[0, 0] = np.nan
    assert not oracle.check_close(nan, ref)[0]


# ---------------------------------------------------------- row reduction

def _exact_row_sums(vals, rows, cols, ldx):
    """Exact rational row sums of fp32 storage (struct-decoded values)."""
    import struct
    from fractions import Fraction
    raw = np.asarray(vals, dtype=np.float32).tobytes()
    dec = struct.unpack(f"<{len(raw) // 4}f", raw)
    return [sum((Fraction(dec[r * ldx + c]) for c in range(cols)), Fraction(0)) for r in range(rows)]


def _reduce_pins_hold(fn):
    """True when ``fn`` (a candidate for oracle.reduce_rows) meets every pin:
    the IREE page's two cases on all-ones input (4096 -> 4096, 4 x 4096 ->
    four 4096s), the arithmetic-series closed form, and exact rational brute
    force on small padded matrices whose padding is NaN."""
    if not np.array_equal(fn(np.ones(4096, np.float32), 1, 4096), [4096.0]):
        return False
    if not np.array_equal(fn(np.ones(4 * 4096, np.float32), 4, 4096), [4096.0] * 4):
        return False
    rows, cols = 3, 1000
    x = (np.arange(cols, dtype=np.float32)[None, :] + np.arange(rows, dtype=np.float32)[:, None] * 7).ravel()
    want = [cols * (cols - 1) / 2 + 7 * r * cols for r in range(rows)]
    if not np.array_equal(fn(x, rows, cols), want):
        return False
    rng = np.random.default_rng(5)
    for rows, cols, pad in [(1, 1, 0), (2, 3, 1), (5, 9, 4), (4, 17, 3), (3, 0, 2)]:
        ldx = cols + pad
        buf = np.full(rows * max(ldx, 1), np.nan, dtype=np.float32)
        for r in range(rows):
            buf[r * ldx:r * ldx + cols] = (rng.standard_normal(cols) * 10.0 ** rng.integers(-3, 4)).astype(np.float32)
        got = fn(buf, rows, cols, ldx)
        exact = _exact_row_sums(buf, rows, cols, ldx)
        for r in range(rows):
            scale = float(sum(abs(float(buf[r * ldx + c])) for c in range(cols)))
            if not np.isfinite(got[r]) or abs(float(exact[r]) - got[r]) > (cols + 1) * 2.0 ** -53 * scale:
                return False
    return True


def test_reduce_rows_pins():
    assert _reduce_pins_hold(oracle.reduce_rows)


def test_reduce_rows_planted_mistakes_are_caught():
    def drop_last(x, rows, cols, ldx=0):
        return oracle.reduce_rows(x, rows, max(cols - 1, 0), ldx or cols)

    def dense_pitch(x, rows, cols, ldx=0):
        return oracle.reduce_rows(x, rows, cols, 0)

    def first_negated(x, rows, cols, ldx=0):
        y = np.array(x, dtype=np.float32, copy=True)
        p = ldx or cols
        for r in range(rows):
            if cols:
                y[r * p] = -y[r * p]
        return oracle.reduce_rows(y, rows, cols, ldx)

    def in_fp32(x, rows, cols, ldx=0):
        p = ldx or cols
        v = np.asarray(x, dtype=np.float32)
        return np.array([np.float32(np.cumsum(v[r * p:r * p + cols], dtype=np.float32)[-1]) if cols else 0.0
                         for r in range(rows)], dtype=np.float64)

    for bad in (drop_last, dense_pitch, first_negated, in_fp32):
        assert not _reduce_pins_hold(bad), bad.__name__


def test_reduce_rows_bound_holds_for_sequential_fp32():
    """The textbook bound for n-term recursive summation, (n - 1) u sum|x|
    (Higham, Accuracy and Stability of Numerical Algorithms, sec. 4.2), is
    what reduce_rows_bound gives for chain = n, depth = 0 (one spare term);
    a plain fp32 left-to-right sum stays inside it, and a sum with one term
    dropped does not."""
    rng = np.random.default_rng(7)
    for n in (10, 1000, 100000):
        x = rng.standard_normal(n).astype(np.float32)
        seq = float(np.cumsum(x, dtype=np.float32)[-1])
        exact = oracle.reduce_rows(x, 1, n)[0]
        bound = oracle.reduce_rows_bound(oracle.reduce_rows_abs(x, 1, n), n, 0)[0]
        assert abs(seq - exact) <= bound
        assert abs(float(np.cumsum(x[:-1], dtype=np.float32)[-1]) - exact) > bound or abs(x[-1]) < bound


# ---------------------------------------------------------------------------
# attention: O = softmax(Q K^T * scale) V per head (the Triton page's second
# dot of Flash Attention, with V contiguous along d)
# ---------------------------------------------------------------------------

def _attn_inputs(heads, sq, sk, d, seed, dtype=oracle.F16):
    case = wl.attn_case(heads, sq, sk, d, dtype)
    return wl.make_attn_inputs(case, seed)


def test_attention_zero_queries_give_the_mean_of_v():
    """Q = 0: every logit is 0, the softmax is uniform, and each output row is
    the mean of V's rows (closed form, independent of the scale)."""
    heads, sq, sk, d = 2, 3, 7, 8
    _, k, v = _attn_inputs(heads, sq, sk, d, seed=1)
    q = torch.zeros(heads * sq * d, dtype=torch.float16)
    o = oracle.attention(q, k, v, heads, sq, sk, d, oracle.F16, scale=0.37)
    vv = oracle.decode(v, oracle.F16).reshape(heads, sk, d)
    for h in range(heads):
        np.testing.assert_allclose(o[h], np.repeat(vv[h].mean(axis=0)[None], sq, axis=0), rtol=0, atol=1e-15)


def test_attention_two_key_closed_form():
    """One query e0, keys a*e0 and 0: logits (a*scale, 0), so
    O = p V0 + (1 - p) V1 with p = 1 / (1 + exp(-a*scale)).  A dropped or
    misplaced scale, or a missing normalisation, fails this."""
    d, a, scale = 4, 3.0, 0.5
    q = torch.zeros(d, dtype=torch.float16)
    q[0] = 1.0
    k = torch.zeros(2 * d, dtype=torch.float16)
    k[0] = a
    v = torch.tensor([1.0, -2.0, 0.5, 4.0, -3.0, 0.25, 2.0, 1.5], dtype=torch.float16)
    o = oracle.attention(q, k, v, 1, 1, 2, d, oracle.F16, scale=scale)
    p = 1.0 / (1.0 + np.exp(-a * scale))
    want = p * np.array([1.0, -2.0, 0.5, 4.0]) + (1 - p) * np.array([-3.0, 0.25, 2.0, 1.5])
    np.testing.assert_allclose(o[0, 0], want, rtol=1e-14, atol=0)
    # the default scale is 1 / sqrt(d)
    o2 = oracle.attention(q, k, v, 1, 1, 2, d, oracle.F16)
    p2 = 1.0 / (1.0 + np.exp(-a / 2.0))
    np.testing.assert_allclose(o2[0, 0], p2 * np.array([1.0, -2.0, 0.5, 4.0]) + (1 - p2) * np.array(
        [-3.0, 0.25, 2.0, 1.5]), rtol=1e-14, atol=0)


def test_attention_rows_sum_to_one_and_key_order_does_not_matter():
    heads, sq, sk, d = 2, 5, 9, 16
    q, k, v = _attn_inputs(heads, sq, sk, d, seed=2)
    ones = torch.ones(heads * sk * d, dtype=torch.float16)
    np.testing.assert_allclose(oracle.attention(q, k, ones, heads, sq, sk, d, oracle.F16), 1.0, rtol=0, atol=1e-14)
    perm = torch.randperm(sk, generator=torch.Generator().manual_seed(3))
    kp = k.reshape(heads, sk, d)[:, perm].reshape(-1)
    vp = v.reshape(heads, sk, d)[:, perm].reshape(-1)
    np.testing.assert_allclose(oracle.attention(q, kp, vp, heads, sq, sk, d, oracle.F16),
                               oracle.attention(q, k, v, heads, sq, sk, d, oracle.F16), rtol=1e-13, atol=1e-15)


def test_attention_composes_from_the_gemm_oracle():
    """The same result through the pinned GEMM oracle: S = Q K^T with K as a
    K-contiguous B operand, then a softmax written out here, then O = P V
    with V as an N-contiguous B operand (the non-TN second dot).  A
    transposed V (or K) fails this."""
    heads, sq, sk, d = 2, 6, 10, 8
    q, k, v = _attn_inputs(heads, sq, sk, d, seed=4)
    scale = 0.3
    o = oracle.attention(q, k, v, heads, sq, sk, d, oracle.F16, scale=scale)
    for h in range(heads):
        qh = q.reshape(heads, sq * d)[h]
        kh = k.reshape(heads, sk * d)[h]
        vh = v.reshape(heads, sk * d)[h]
        s = oracle.gemm(sq, sk, d, qh, oracle.K_CONTIG, d, oracle.F16, kh, oracle.K_CONTIG, d, oracle.F16) * scale
        e = np.exp(s - s.max(axis=1, keepdims=True))
        p = e / e.sum(axis=1, keepdims=True)
        pv = np.zeros((sq, d))
        vv = oracle.b_logical(vh, sk, d, oracle.MN_CONTIG, d, oracle.F16)
        for j in range(sk):
            pv += p[:, j:j + 1] * vv[j:j + 1, :]
        np.testing.assert_allclose(o[h], pv, rtol=1e-13, atol=1e-15)


def test_attention_rows_match_full():
    heads, sq, sk, d = 3, 7, 11, 16
    q, k, v = _attn_inputs(heads, sq, sk, d, seed=5, dtype=oracle.BF16)
    full = oracle.attention(q, k, v, heads, sq, sk, d, oracle.BF16)
    hs, rs = [0, 2, 1, 2], [0, 6, 3, 1]
    np.testing.assert_allclose(oracle.attention_rows(hs, rs, q, k, v, heads, sq, sk, d, oracle.BF16),
                               full[hs, rs], rtol=1e-13, atol=1e-15)


def test_planted_attention_mistake_is_caught(monkeypatch):
    """A softmax normalised over the wrong axis must fail the pins above."""
    def wrong_axis(s):
        e = np.exp(s - s.max())
        return e / e.sum(axis=0, keepdims=True)
    monkeypatch.setattr(oracle, "_softmax_rows", wrong_axis)
    with pytest.raises(AssertionError):
        test_attention_rows_sum_to_one_and_key_order_does_not_matter()
