"""Pins of the CPU oracle against facts outside the oracle itself.

Each test ties one part of the method, as the mmaemu v0.1 documentation states
it, to a library routine, a closed form, an invariant or brute force, so that a
plausible mistake in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong rounding) fails at least one of them.
"""
import ctypes
import math
import platform
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import spec

FMTS = ("e4m3fn", "e5m2")
TORCH_FP8 = {"e4m3fn": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
PAIRS = (("e4m3fn", "e4m3fn"), ("e4m3fn", "e5m2"), ("e5m2", "e4m3fn"), ("e5m2", "e5m2"))


def f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def bits32(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def finite_codes(fmt):
    """all finite codes of a format"""
    out = []
    for c in range(256):
        if fmt == "e4m3fn" and (c & 0x7F) == 0x7F:
            continue
        if fmt == "e5m2" and ((c >> 2) & 31) == 31:
            continue
        out.append(c)
    return np.array(out, dtype=np.uint8)


def normal_codes(fmt):
    fb = 3 if fmt == "e4m3fn" else 2
    return np.array([c for c in finite_codes(fmt) if (c & 0x7F) >> fb != 0], dtype=np.uint8)


def code_value(fmt, code):
    """decoded value through torch's fp8 -> fp32 conversion (library routine)"""
    t = torch.tensor([code], dtype=torch.uint8).view(TORCH_FP8[fmt]).to(torch.float32)
    return float(t.item())


# ---------------------------------------------------------------------------
# decode: exhaustive against torch's FP8 conversion
# ("Validation evidence", claims table: subnormal inputs keep exponent emin)
@pytest.mark.parametrize("fmt", FMTS)
def test_decode_exhaustive_vs_torch(orc, fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    bias = 7 if fmt == "e4m3fn" else 15
    for c in range(256):
        nan, inf, neg, sig, e, f = orc.decode(fmt, c)
        r = ref[c]
        if math.isnan(r):
            assert nan == 1 and inf == 0
            continue
        if math.isinf(r):
            assert inf == 1 and nan == 0 and neg == (r < 0)
            continue
        assert nan == 0 and inf == 0
        assert (-1) ** neg * sig * 2.0 ** (e - f) == r
        if r != 0:
            if sig >= 2 ** f:                          # normal code: e = floor(log2 |v|)
                assert e == math.floor(math.log2(abs(r)))
            else:                                      # subnormal code keeps emin
                assert e == 1 - bias
        assert neg == (c >> 7)


# products: all 65,536 code pairs per format pair, exact value and label
@pytest.mark.parametrize("fa,fb", PAIRS)
def test_products_exhaustive(orc, fa, fb):
    ca = finite_codes(fa)
    cb = finite_codes(fb)
    A, B = np.meshgrid(ca, cb, indexing="ij")
    A = A.ravel()
    B = B.ravel()
    p = orc.products(A, fa, B, fb)
    va = torch.tensor(A).view(TORCH_FP8[fa]).to(torch.float64).numpy()
    vb = torch.tensor(B).view(TORCH_FP8[fb]).to(torch.float64).numpy()
    want = va * vb                                      # exact in binary64 (<= 8 bits)
    got = np.where(p[:, 0] == 1, -1.0, 1.0) * p[:, 1] * np.exp2(p[:, 2] - p[:, 3])
    nz = want != 0
    assert np.array_equal(got[nz], want[nz])
    assert np.all(p[~nz, 1] == 0)
    la = np.array([orc.decode(fa, int(c))[4] for c in range(256)])
    lb = np.array([orc.decode(fb, int(c))[4] for c in range(256)])
    assert np.array_equal(p[:, 2], la[A] + lb[B])       # label exponent e_a + e_b
    assert np.array_equal(p[:, 0], (A >> 7) ^ (B >> 7))  # sign


# ---------------------------------------------------------------------------
# blk with all-zero products: closed form, c truncated to F+1 = 14 significant
# bits ("an all-zero block still truncates c"; zeros are +0).  For finite c the
# truncation toward zero to 14 significant bits clears the low 10 fraction bits,
# for normal and subnormal c alike (subnormal grid 2^(-126-13)).
@pytest.mark.parametrize("B", (32, 16))
def test_blk_zero_products_closed_form(orc, B):
    rng = np.random.default_rng(1)
    exps = np.repeat(np.arange(0, 255, dtype=np.uint32), 1024)
    mants = rng.integers(0, 1 << 23, exps.size, dtype=np.uint32)
    mants[::1024] = 0
    mants[1::1024] = (1 << 23) - 1
    mants[2::1024] = 0x3FF
    mants[3::1024] = 0x400
    signs = rng.integers(0, 2, exps.size, dtype=np.uint32) << 31
    c = signs | (exps << 23) | mants
    zcodes = rng.choice(np.array([0x00, 0x80], dtype=np.uint8), size=(c.size, B))
    got = orc.blk_many(c, zcodes, "e4m3fn", zcodes[:, ::-1].copy(), "e4m3fn", F=13)
    want = (c & 0xFFFFFC00).astype(np.uint32)
    want[(want & 0x7FFFFFFF) == 0] = 0          # truncated to zero -> +0
    assert np.array_equal(got, want)
    # every fraction pattern of the (negative) subnormal and the smallest normal
    # binade, with one zero product per block
    full = np.arange(1 << 23, dtype=np.uint32)
    c = np.concatenate([full | (1 << 31), full | (1 << 23)])
    z = np.full((c.size, 1), 0x80 if B == 32 else 0x00, np.uint8)
    got = orc.blk_many(c, z, "e4m3fn", z, "e4m3fn", F=13)
    want = (c & 0xFFFFFC00).astype(np.uint32)
    want[(want & 0x7FFFFFFF) == 0] = 0
    assert np.array_equal(got, want)


# blk, products of one label exponent: every term lies on the grid, so the block
# returns the exact sum (when below 2^(E+1)), or the exact sum truncated to 14
# significant bits (carry).  Exact sums by Fraction.
@pytest.mark.parametrize("fa,fb", PAIRS[:3])
def test_blk_shared_exponent_exact(orc, fa, fb):
    rng = np.random.default_rng(2)
    fba = 3 if fa == "e4m3fn" else 2
    fbb = 3 if fb == "e4m3fn" else 2
    n_ok = n_carry = 0
    for trial in range(3000):
        n = int(rng.integers(1, 33))
        Ea = int(rng.integers(1, 15 if fa == "e4m3fn" else 30))
        Eb = int(rng.integers(1, 15 if fb == "e4m3fn" else 30))
        ma = rng.integers(0, 1 << fba, n)
        mb = rng.integers(0, 1 << fbb, n)
        sa = rng.integers(0, 2, n) << 7
        sb = rng.integers(0, 2, n) << 7
        a = (sa | (Ea << fba) | ma).astype(np.uint8)
        b = (sb | (Eb << fbb) | mb).astype(np.uint8)
        if fa == "e4m3fn":
            a[(a & 0x7F) == 0x7F] ^= 1          # keep clear of the NaN code
        if fb == "e4m3fn":
            b[(b & 0x7F) == 0x7F] ^= 1
        exact = sum(Fraction(code_value(fa, int(x))) * Fraction(code_value(fb, int(y)))
                    for x, y in zip(a, b))
        got = orc.blk_many(np.zeros(1, np.uint32), a[None, :], fa, b[None, :], fb, F=13)[0]
        got_v = Fraction(float(f32(got)))
        E = Ea - (7 if fa == "e4m3fn" else 15) + Eb - (7 if fb == "e4m3fn" else 15)
        if exact == 0:
            assert got == 0
            continue
        if abs(exact) < Fraction(2) ** (E + 1):
            assert got_v == exact
            n_ok += 1
        else:                                   # carry: 14 significant bits, toward zero
            g = Fraction(2) ** (E - 13)
            S = abs(exact) / g
            assert S.denominator == 1
            S = S.numerator
            L = S.bit_length()
            S = (S >> (L - 14)) << (L - 14)
            assert got_v == (1 if exact > 0 else -1) * S * g
            n_carry += 1
    assert n_ok > 100 and n_carry > 100


# a block whose result is exactly zero, or whose truncated terms cancel while the
# exact sum does not, returns +0 ("Validation evidence", Scope table, Ada row)
def test_blk_zero_results_are_plus_zero(orc):
    # p and -p
    a = np.array([[0x50, 0xD0]], dtype=np.uint8)       # +x, -x (e4m3)
    b = np.array([[0x48, 0x48]], dtype=np.uint8)
    assert orc.blk_many(np.zeros(1, np.uint32), a, "e4m3fn", b, "e4m3fn")[0] == 0
    # +A, -A and a negative product far below the grid: the exact sum is negative,
    # the truncated sum is zero -> +0, not -0
    a = np.array([[0x70, 0xF0, 0x81]], dtype=np.uint8)  # 128, -128, -2^-9
    b = np.array([[0x70, 0x70, 0x01]], dtype=np.uint8)  # 128, 128, 2^-9
    r = orc.blk_many(np.zeros(1, np.uint32), a, "e4m3fn", b, "e4m3fn")[0]
    assert r == 0
    ok, S, E = orc.blk_exact(0, a[0], "e4m3fn", b[0], "e4m3fn", 13)
    assert ok and S == 0 and E == 14
    # c cancelled by a product: c = -(product) exactly
    c = bits32(np.float32(-16384.0))
    r = orc.blk_many(np.array([c], np.uint32), np.array([[0x70]], np.uint8), "e4m3fn",
                     np.array([[0x70]], np.uint8), "e4m3fn")[0]
    assert r == 0
    # all-zero block with c = -0 -> +0
    r = orc.blk_many(np.array([0x80000000], np.uint32), np.array([[0x80] * 32], np.uint8),
                     "e4m3fn", np.array([[0x00] * 32], np.uint8), "e4m3fn")[0]
    assert r == 0


# library special case: one product per block (B=1) with F=23 and operands of one
# sign is fp32 addition rounded toward zero.  Proof sketch: with normal FP8
# operands, max(|c|, |p|) >= 2^E, so the rounding grid of c + p is g = 2^(E-23)
# or coarser; the one term below the grid loses only bits that toward-zero
# rounding of the sum also drops.  Checked against the host FPU under
# fesetround(FE_TOWARDZERO).
def _fesetround():
    libm = ctypes.CDLL("libm.so.6")
    mach = platform.machine()
    if mach in ("x86_64", "AMD64"):
        return libm, 0x000, 0xC00
    if mach in ("aarch64", "arm64"):
        return libm, 0x000000, 0xC00000
    pytest.skip(f"unknown rounding-mode constants on {mach}")


def test_blk_single_product_is_fp32_rz_addition(orc):
    libm, FE_TONEAREST, FE_TOWARDZERO = _fesetround()
    rng = np.random.default_rng(3)
    for fa, fb in PAIRS[:3]:
        na, nb = normal_codes(fa), normal_codes(fb)
        n = 60000
        a = rng.choice(na, n)
        b = rng.choice(nb, n)
        same = ((a >> 7) ^ (b >> 7)) & 1
        va = torch.tensor(a).view(TORCH_FP8[fa]).to(torch.float64).numpy()
        vb = torch.tensor(b).view(TORCH_FP8[fb]).to(torch.float64).numpy()
        p = (va * vb).astype(np.float32)               # exact
        # c of the product's sign: near the product's magnitude, far below, far above,
        # subnormal and zero
        scale = np.exp2(rng.integers(-30, 30, n)).astype(np.float64)
        cmag = np.abs(p.astype(np.float64)) * scale * rng.uniform(0.5, 2.0, n)
        cmag[::7] = 0.0
        cmag[1::7] = rng.uniform(0, 1, n)[1::7] * 1e-39
        c = (cmag * np.where(same == 1, -1.0, 1.0)).astype(np.float32)
        cb = bits32(c)
        got = orc.blk_many(cb, a[:, None], fa, b[:, None], fb, F=23)
        old = libm.fegetround()
        try:
            assert libm.fesetround(FE_TOWARDZERO) == 0
            probe = np.float32(1.0) + np.float32(0.99999994)
            if probe == np.float32(2.0):
                pytest.skip("numpy does not honour the dynamic rounding mode here")
            want = bits32(c + p)
        finally:
            libm.fesetround(old)
        # a zero sum of c = -0 and p = 0 cannot occur (normal codes); +0 + p = p
        assert np.array_equal(got, want), (fa, fb, np.flatnonzero(got != want)[:5])


# large F: with F = 60 no term of a 32-product block falls below the grid, so the
# exact block sum S * 2^(E-60) equals the exact sum of the products (Fraction)
@pytest.mark.parametrize("fa,fb", PAIRS)
def test_blk_large_F_is_exact_sum(orc, fa, fb):
    rng = np.random.default_rng(4)
    ca, cb = finite_codes(fa), finite_codes(fb)
    for _ in range(400):
        n = int(rng.integers(1, 33))
        a = rng.choice(ca, n)
        b = rng.choice(cb, n)
        ok, S, E = orc.blk_exact(0, a, fa, b, fb, 60)
        exact = sum(Fraction(code_value(fa, int(x))) * Fraction(code_value(fb, int(y)))
                    for x, y in zip(a, b))
        nonzero = [(int(x), int(y)) for x, y in zip(a, b)
                   if code_value(fa, int(x)) * code_value(fb, int(y)) != 0]
        if not nonzero:
            assert not ok
            continue
        assert ok
        assert Fraction(S) * Fraction(2) ** (E - 60) == exact
        labels = [orc.decode(fa, x)[4] + orc.decode(fb, y)[4] for x, y in nonzero]
        assert E == max(labels)


# ---------------------------------------------------------------------------
# brute force: the C oracle against the independent Fraction model on random and
# adversarial blocks (subnormals, +-max, carries, cancellation) and chains
def _adversarial_codes(rng, fmt, n):
    fc = finite_codes(fmt)
    fb = 3 if fmt == "e4m3fn" else 2
    mx = 0x7E if fmt == "e4m3fn" else 0x7B
    pool = np.concatenate([fc, np.array([0, 0x80, mx, mx | 0x80], np.uint8).repeat(16),
                           np.arange(1, 1 << fb, dtype=np.uint8).repeat(8)])
    return rng.choice(pool, n)


@pytest.mark.parametrize("fa,fb", PAIRS[:3])
@pytest.mark.parametrize("B", (32, 16))
def test_blk_c_oracle_vs_fraction_model(orc, fa, fb, B):
    rng = np.random.default_rng(5 + B)
    count = 2500
    a = _adversarial_codes(rng, fa, (count, B))
    b = _adversarial_codes(rng, fb, (count, B))
    cvals = np.concatenate([
        rng.normal(0, 1, count // 4) * np.exp2(rng.integers(-20, 40, count // 4)),
        np.zeros(count // 4),
        rng.normal(0, 1, count // 4) * 1e-3,
        rng.normal(0, 1, count - 3 * (count // 4)) * 1e6])
    cb = bits32(cvals.astype(np.float32))
    cb[::50] = rng.integers(1, 1 << 23, cb[::50].size, dtype=np.uint32)   # fp32 subnormals
    got = orc.blk_many(cb, a, fa, b, fb, F=13)
    for j in range(count):
        terms = []
        for x, y in zip(a[j], b[j]):
            _, va, la = spec.decode(fa, int(x))
            _, vb, lb = spec.decode(fb, int(y))
            terms.append((va * vb, la + lb))
        want = spec.blk(spec.f32_value(int(cb[j])), terms, 13)
        assert got[j] == spec.f32_bits(want), j


@pytest.mark.parametrize("preset", ("hopper", "ada"))
def test_gemm_c_oracle_vs_fraction_model(orc, preset):
    rng = np.random.default_rng(11)
    for trial in range(40):
        fa, fb = PAIRS[trial % 3]
        M, N = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        K = int(rng.choice([16, 48, 128, 144, 256, 400]))
        a = _adversarial_codes(rng, fa, (M, K))
        b = _adversarial_codes(rng, fb, (N, K))
        fast = bool(trial % 2)
        S = int(rng.choice([1, 2, 3, 5]))
        pairwise = preset == "ada" and trial % 4 == 3
        P = dict(orc.PRESETS[preset])
        P["combine"] = int(pairwise)
        idx_m, idx_n = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        got = orc.acc_sampled(a, b, fa, fb, idx_m.ravel(), idx_n.ravel(), fast, S, P)
        for i, (m, n) in enumerate(zip(idx_m.ravel(), idx_n.ravel())):
            want = spec.accumulator(a[m], b[n], fa, fb, fast, S, preset, pairwise)
            assert got[i] == spec.f32_bits(want), (trial, m, n)
        for od in ("f32", "bf16", "f16"):
            full = orc.scaled_mm(a, b, fa, fb, 1 / 64, 1 / 32, od, fast, S, P)
            for i, (m, n) in enumerate(zip(idx_m.ravel(), idx_n.ravel())):
                want = spec.accumulator(a[m], b[n], fa, fb, fast, S, preset, pairwise)
                assert full[m, n] == spec.epilogue(want, 1 / 64, 1 / 32, od)


# ---------------------------------------------------------------------------
# slow accumulation ("Validation evidence", H100 probe: restart every 128 and add
# in K order)
def test_slow_equals_fast_when_restart_covers_chain(orc):
    rng = np.random.default_rng(12)
    for _ in range(50):
        K = int(rng.choice([32, 96, 256]))
        a = _adversarial_codes(rng, "e4m3fn", K)
        b = _adversarial_codes(rng, "e4m3fn", K)
        assert orc.chain(a, "e4m3fn", b, "e4m3fn", False, 32, 13, 4096) == \
            orc.chain(a, "e4m3fn", b, "e4m3fn", True, 32, 13, 4096)


def test_slow_is_k_order_fp32_sum_of_128_chunks(orc):
    rng = np.random.default_rng(13)
    for _ in range(200):
        K = 384
        a = _adversarial_codes(rng, "e4m3fn", K)
        b = _adversarial_codes(rng, "e4m3fn", K)
        parts = [orc.chain(a[j:j + 128], "e4m3fn", b[j:j + 128], "e4m3fn", True)
                 for j in range(0, K, 128)]
        p = f32(np.array(parts, np.uint32))
        want = bits32((p[0] + p[1]) + p[2])            # numpy fp32, round to nearest
        assert orc.chain(a, "e4m3fn", b, "e4m3fn", False) == want


# ---------------------------------------------------------------------------
# split-K
def test_split_index_rules(orc):
    # contiguous: ceil(T/S) tiles per split, trailing splits empty
    K = 262144
    T = K // 128
    got = [orc.split_indices(K, 24, 0, 128, s) for s in range(24)]
    assert [len(g) // 128 for g in got] == [86] * 23 + [T - 86 * 23]
    assert np.array_equal(np.concatenate(got), np.arange(K))
    got = [orc.split_indices(256, 3, 0, 128, s) for s in range(3)]
    assert [len(g) for g in got] == [128, 128, 0]
    # interleaved: 64-wide tiles dealt round-robin
    for S in (2, 3, 8):
        K = 64 * 11 + 16
        seen = np.zeros(K, int)
        for s in range(S):
            idx = orc.split_indices(K, S, 1, 64, s)
            assert np.all(np.diff(idx) > 0)
            assert np.all((idx // 64) % S == s)
            seen[idx] += 1
        assert np.all(seen == 1)


def test_split_invariants(orc):
    rng = np.random.default_rng(14)
    M, N, K = 2, 3, 1024
    a = _adversarial_codes(rng, "e4m3fn", (M, K))
    b = _adversarial_codes(rng, "e4m3fn", (N, K))
    im, jn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    im, jn = im.ravel(), jn.ravel()
    acc = lambda fast, S, preset="hopper": orc.acc_sampled(a, b, "e4m3fn", "e4m3fn", im, jn, fast, S, preset)
    # hopper, slow, one 128-tile per split == unsplit slow (same K-order sum)
    assert np.array_equal(acc(False, K // 128), acc(False, 1))
    # fast, one tile per split: the serial fp32 sum of independent 128-chains
    want = []
    for m, n in zip(im, jn):
        parts = f32(np.array([orc.chain(a[m, j:j + 128], "e4m3fn", b[n, j:j + 128], "e4m3fn", True)
                              for j in range(0, K, 128)], np.uint32))
        s = parts[0]
        for p in parts[1:]:
            s = np.float32(s + p)
        want.append(bits32(s))
    assert np.array_equal(acc(True, K // 128), np.array(want, np.uint32))
    # an empty contiguous split adds +0: K=256 with S=3 equals S=2
    a2, b2 = a[:, :256].copy(), b[:, :256].copy()
    r3 = orc.acc_sampled(a2, b2, "e4m3fn", "e4m3fn", im, jn, True, 3)
    r2 = orc.acc_sampled(a2, b2, "e4m3fn", "e4m3fn", im, jn, True, 2)
    assert np.array_equal(r3, r2)
    # ada interleaved, one-hot tile: only the owning split sees nonzero products
    K = 64 * 6
    a3 = np.zeros((1, K), np.uint8)
    b3 = _adversarial_codes(rng, "e4m3fn", (1, K))
    a3[0, 64 * 3:64 * 4] = _adversarial_codes(rng, "e4m3fn", 64)
    full = orc.acc_sampled(a3, b3, "e4m3fn", "e4m3fn", [0], [0], True, 2, "ada")[0]
    tile = orc.chain(a3[0, 192:256], "e4m3fn", b3[0, 192:256], "e4m3fn", True, 16, 13, 128)
    assert full == tile


# combination order ("Validation evidence", claims: S = 3 pairwise is (p2+p0)+p1)
def test_combine_orders(orc):
    p = np.array([2.0 ** 24, 1.0, -2.0 ** 24], np.float32)
    pb = bits32(p)
    serial = bits32(np.float32(np.float32(p[0] + p[1]) + p[2]))
    pairwise = bits32(np.float32(np.float32(p[2] + p[0]) + p[1]))
    assert serial != pairwise
    assert orc.combine(pb, False) == serial
    assert orc.combine(pb, True) == pairwise
    rng = np.random.default_rng(15)
    for S in (2, 4, 8, 24):
        x = (rng.normal(size=S) * np.exp2(rng.integers(-10, 30, S))).astype(np.float32)
        s = x[0]
        for v in x[1:]:
            s = np.float32(s + v)
        assert orc.combine(bits32(x), False) == bits32(s)


# ---------------------------------------------------------------------------
# epilogue ("Limitations", corrections: y = fma(acc, alpha, +0); claims: bf16/fp16
# rounded from the fp32 value)
def _special_f32(rng, n):
    x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    specials = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF,
                         0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x3F800000, 0xBF800000,
                         0x33800000, 0x39000000, 0x00000010], np.uint32)
    x[:specials.size] = specials
    return x


def test_fp32_arithmetic_vs_host(orc):
    rng = np.random.default_rng(16)
    n = 400000
    a = _special_f32(rng, n)
    b = rng.permutation(_special_f32(rng, n))
    # exponent-close pairs, where rounding and cancellation matter
    b[: n // 2] = (a[: n // 2] & 0xFF800000) | rng.integers(0, 1 << 23, n // 2, dtype=np.uint32)
    b[: n // 4] ^= 0x80000000
    with np.errstate(all="ignore"):
        fa, fb = f32(a), f32(b)
        add = bits32(fa + fb)
        mul = bits32(fa * fb)
        prod = fa.astype(np.float64) * fb.astype(np.float64)   # exact
        fma = bits32(np.where(prod == 0, np.float32(0.0), prod.astype(np.float32)))
    canon = lambda v: np.where(np.isnan(f32(v)), np.uint32(0x7FC00000), v)
    assert np.array_equal(orc.f32_add_rn(a, b), canon(add))
    assert np.array_equal(orc.f32_mul_rn(a, b), canon(mul))
    assert np.array_equal(orc.f32_fma_plus0(a, b), canon(fma))


def test_bf16_fp16_rounding_vs_library(orc):
    rng = np.random.default_rng(17)
    x = _special_f32(rng, 500000)
    # ties and near-ties of bf16: low 16 bits 0x8000 / 0x7FFF / 0x8001
    x[1000:2000] = (x[1000:2000] & 0xFFFF0000) | 0x8000
    x[2000:3000] = (x[2000:3000] & 0xFFFF0000) | 0x7FFF
    x[3000:4000] = (x[3000:4000] & 0xFFFF0000) | 0x8001
    t = torch.from_numpy(x.view(np.int32).copy()).view(torch.float32)
    bf = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bf = np.where(np.isnan(f32(x)), np.uint16(0x7FC0), bf)
    assert np.array_equal(orc.f32_to_bf16(x), bf)
    with np.errstate(all="ignore"):
        h = f32(x).astype(np.float16).view(np.uint16)
    h = np.where(np.isnan(f32(x)), np.uint16(0x7E00), h)
    assert np.array_equal(orc.f32_to_f16(x), h)


def test_epilogue_double_rounding_and_zero_sign(orc):
    rng = np.random.default_rng(18)
    # accumulators whose exact product with alpha lies just beside a bf16 tie: the
    # fp32 rounding moves it onto the tie and bf16 then rounds to even
    n = 20000
    acc = np.zeros(n, np.float32)
    alpha = np.float32(3.0)
    base = rng.integers(0x3F800000, 0x4F000000, n, dtype=np.uint32) & 0xFFFF0000
    for i in range(n):
        hb = f32(np.uint32(base[i] | 0x8000))          # an exact bf16 tie in fp32
        acc[i] = np.float32(np.float64(hb) / 3.0)
    ab = bits32(acc)
    y = bits32((acc.astype(np.float64) * np.float64(alpha)).astype(np.float32))
    t = torch.from_numpy(y.view(np.int32).copy()).view(torch.float32)
    want = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.epilogue(ab, 1.5, 2.0, "bf16")
    assert np.array_equal(got, want)
    # a single rounding of the exact product to 8 significant bits would differ
    # on some of them (round-half-even on the exact binary64 value)
    def single_bf16(v):
        m, e = math.frexp(v)
        return math.ldexp(round(m * 256.0), e - 8)
    want_v = torch.from_numpy(want.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    differ = sum(single_bf16(float(x) * 3.0) != w for x, w in zip(acc, want_v))
    assert differ > 100
    # zero sign: +0 for an exactly zero product, the sign kept on underflow
    acc = bits32(np.array([0.0, 1e-30, -1e-30, 1.0, -1.0, 0.0], np.float32))
    for sa, sb in ((1.0, -1.0), (0.0, 1.0), (-0.0, 1.0), (1e-30, 1e-20), (-1e-30, 1e-20)):
        got = orc.epilogue(acc, sa, sb, "f32")
        alpha = np.float32(sa) * np.float32(sb)
        prod = f32(acc).astype(np.float64) * np.float64(alpha)
        want = bits32(np.where(prod == 0, np.float32(0.0), prod.astype(np.float32)))
        assert np.array_equal(got, want), (sa, sb)
    # power-of-two alpha scales exactly
    accs = (rng.normal(size=1000) * 1e6).astype(np.float32)
    got = orc.epilogue(bits32(accs), 1 / 64, 1 / 32, "f32")
    assert np.array_equal(f32(got), accs * np.float32(2.0 ** -11))


# ---------------------------------------------------------------------------
# NaN rule ("Limitations", corrections): a NaN code anywhere in row m of A or
# column n of B makes output (m, n) the canonical NaN; nothing else is NaN
@pytest.mark.parametrize("fmt", FMTS)
def test_nan_rule(orc, fmt):
    rng = np.random.default_rng(19)
    M, N, K = 5, 7, 96
    a = rng.choice(finite_codes(fmt), (M, K))
    b = rng.choice(finite_codes("e4m3fn"), (N, K))
    nan = 0x7F if fmt == "e4m3fn" else 0x7E
    a[2, 17] = nan
    b[4, 90] = 0xFF
    out = orc.scaled_mm(a, b, fmt, "e4m3fn", 1.0, 1.0, "f32", False, 2)
    isnan = out == 0x7FC00000
    want = np.zeros((M, N), bool)
    want[2, :] = True
    want[:, 4] = True
    assert np.array_equal(isnan, want)
    assert not np.any(np.isnan(f32(out[~want])))


# Inf codes (E5M2): the IEEE reading, checked against a float64 dot product of
# the decoded values (library IEEE arithmetic decides NaN vs +-Inf)
def test_inf_reading_vs_ieee_dot(orc):
    rng = np.random.default_rng(20)
    M, N, K = 12, 12, 64
    for trial in range(30):
        a = rng.choice(finite_codes("e5m2"), (M, K))
        b = rng.choice(finite_codes("e4m3fn"), (N, K))
        for _ in range(4):
            a[rng.integers(M), rng.integers(K)] = rng.choice([0x7C, 0xFC])
        b[rng.integers(N), rng.integers(K)] = 0x00
        b[:, 5] = 0x00
        out = orc.scaled_mm(a, b, "e5m2", "e4m3fn", 1.0, 1.0, "f32", True, 1)
        va = torch.tensor(a).view(torch.float8_e5m2).to(torch.float64).numpy()
        vb = torch.tensor(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        with np.errstate(all="ignore"):
            ref = va @ vb.T
        o = f32(out)
        nonfinite = ~np.isfinite(ref)
        assert np.array_equal(np.isnan(o), np.isnan(ref))
        assert np.array_equal(np.isinf(o) & (o > 0), np.isposinf(ref))
        assert np.array_equal(np.isinf(o) & (o < 0), np.isneginf(ref))
        assert not np.any(~np.isfinite(o[~nonfinite]))


# rounding helper against numpy conversions of exact binary64 values
def test_round_helper_vs_numpy(orc):
    rng = np.random.default_rng(21)
    for _ in range(20000):
        mag = int(rng.integers(1, 1 << 53, dtype=np.uint64))
        exp2 = int(rng.integers(-220, 80))
        v = math.ldexp(float(mag), exp2)
        if v == 0 or math.isinf(v) or Fraction(v) != Fraction(mag) * Fraction(2) ** exp2:
            continue
        neg = int(rng.integers(0, 2))
        with np.errstate(all="ignore"):
            want32 = int(np.array([-v if neg else v], np.float64).astype(np.float32).view(np.uint32)[0])
            want16 = int(np.array([-v if neg else v], np.float64).astype(np.float16).view(np.uint16)[0])
        assert orc.round_bits(neg, mag, exp2, 0, 0) == want32
        assert orc.round_bits(neg, mag, exp2, 2, 0) == want16


# fp8 output ("Validation evidence", claims table: scale_result is a separate fp32
# multiply before saturation to the format's maximum): round to nearest even into
# the format, saturate to +-max (Inf too), NaN -> 0x7F.  Against torch's fp8 cast
# of the value clamped to +-max (which rounds to nearest even).
@pytest.mark.parametrize("fmt", FMTS)
def test_f32_to_fp8_saturating_vs_torch(orc, fmt):
    rng = np.random.default_rng(22)
    mx = 448.0 if fmt == "e4m3fn" else 57344.0
    x = _special_f32(rng, 300000)
    # values near the format's range: ties, midpoints, near max and subnormals
    near = (rng.normal(size=100000) * mx * np.exp2(rng.integers(-20, 3, 100000))).astype(np.float32)
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(TORCH_FP8[fmt]).to(torch.float32).numpy()
    vals = vals[np.isfinite(vals)]
    mids = ((vals[:, None] + vals[None, :]) / 2).astype(np.float32).ravel()
    x = np.concatenate([x, bits32(near), bits32(mids), bits32(vals)])
    got = orc.f32_to_fp8(x, fmt)
    xf = torch.from_numpy(f32(x).copy()).clamp(-mx, mx)
    want = xf.to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    want = np.where(np.isnan(f32(x)), np.uint8(0x7F), want)
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:10]


def test_fp8_output_epilogue_rounds_scale_result_separately(orc):
    rng = np.random.default_rng(23)
    acc = (rng.normal(size=50000) * np.exp2(rng.integers(-10, 20, 50000))).astype(np.float32)
    for sa, sb, sr in ((1 / 64, 1 / 32, 3.0), (0.7, 1.3, 0.11), (1.0, 1.0, 1e-30), (2.0, 3.0, -5.0)):
        for fmt in FMTS:
            got = orc.epilogue(bits32(acc), sa, sb, fmt, scale_result=sr)
            alpha = np.float32(sa) * np.float32(sb)
            prod = acc.astype(np.float64) * np.float64(alpha)
            y = np.where(prod == 0, np.float32(0.0), prod.astype(np.float32))
            z = (y * np.float32(sr)).astype(np.float32)              # separate fp32 multiply
            mx = 448.0 if fmt == "e4m3fn" else 57344.0
            want = torch.from_numpy(z.copy()).clamp(-mx, mx).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
            want = np.where(np.isnan(z), np.uint8(0x7F), want)
            assert np.array_equal(got, want), (sa, sb, sr, fmt)
    # near FP8 rounding midpoints, where rounding y first and then multiplying by
    # scale_result differs from one rounding of acc * RN(alpha * scale_result): the
    # accumulators within 8 ulps of each midpoint / (alpha * sr)
    for fmt in FMTS:
        vals = torch.arange(256, dtype=torch.uint8).view(TORCH_FP8[fmt]).float().numpy()
        vals = np.unique(vals[np.isfinite(vals) & (vals > 0)])
        mids = (vals[:-1] + vals[1:]) / 2
        mx = 448.0 if fmt == "e4m3fn" else 57344.0
        for sa, sb, sr in ((0.7, 1.3, 3.0), (0.3, 0.9, 5.0), (1.1, 0.37, 0.3)):
            alpha = np.float32(np.float32(sa) * np.float32(sb))
            base = (mids / (np.float64(alpha) * np.float64(np.float32(sr)))).astype(np.float32)
            near = (base.view(np.int32)[:, None] + np.arange(-8, 9, dtype=np.int32)[None, :])
            accm = np.concatenate([near.ravel(), (near.ravel() | np.int32(-2**31))]).view(np.float32)
            y = (accm.astype(np.float64) * np.float64(alpha)).astype(np.float32)
            z = (y.astype(np.float64) * np.float64(np.float32(sr))).astype(np.float32)
            want = torch.from_numpy(z.copy()).clamp(-mx, mx).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
            one = (accm.astype(np.float64) *
                   np.float64(np.float32(np.float64(alpha) * np.float64(np.float32(sr))))).astype(np.float32)
            assert (torch.from_numpy(one.copy()).clamp(-mx, mx).to(TORCH_FP8[fmt]).view(torch.uint8)
                    .numpy() != want).sum() > 0     # the cases do separate the two readings
            got = orc.epilogue(bits32(accm), sa, sb, fmt, scale_result=sr)
            assert np.array_equal(got, want), (sa, sb, sr, fmt)
    # without scale_result: the fp32 y converts directly
    got = orc.epilogue(bits32(acc), 1.0, 1.0, "e4m3fn")
    want = torch.from_numpy(acc.copy()).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


# The presets against the constants the pages state (tests/golden/page_constants.json,
# each entry citing its page and table), and the one combine order they print.
def test_presets_and_pairwise_order_match_the_pages(orc):
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_constants.json")
    golden = json.load(open(path))
    for name in ("hopper", "ada"):
        want = {k: v["value"] for k, v in golden[name].items()}
        assert orc.PRESETS[name] == want, name
    assert golden["pairwise_S3_order"]["value"] == "(p2 + p0) + p1"
    # S = 3 pairwise: (p2 + p0) + p1 in fp32 round to nearest even, which here differs
    # from the serial (p0 + p1) + p2
    p = np.array([1.0, -1.0, 2.0 ** -30], dtype=np.float32)
    pairwise = np.float32(np.float32(p[2] + p[0]) + p[1])
    serial = np.float32(np.float32(p[0] + p[1]) + p[2])
    assert pairwise != serial
    assert orc.combine(bits32(p), True) == int(bits32(np.array([pairwise]))[0])
    assert orc.combine(bits32(p), False) == int(bits32(np.array([serial]))[0])
