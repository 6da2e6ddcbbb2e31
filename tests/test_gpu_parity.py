"""GPU parity: the CUDA path (C ABI through the package binding) against the CPU
oracle, bit for bit, on every workload -- at oracle-sized shapes that span several
CTA tiles with ragged tails (full comparison), and at the full sizes in the
configuration the benchmark times (sampled outputs, computed one by one by the
oracle) -- plus the edge and degenerate cases."""
import numpy as np
import pytest
import torch

from bit_exact_fp8_gb300 import workloads as W
from helpers import (assert_bits_equal, gpu_run, oracle_full, oracle_sampled,
                     sample_indices)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def full_check(cs, **kw):
    a, b = W.make_inputs(cs)
    got = gpu_run(cs, a, b, **kw)
    want = oracle_full(cs, a, b, preset=kw.get("preset"))
    assert_bits_equal(got, want, cs.name)


def sampled_check(cs, count=256):
    a, b = W.make_inputs(cs)
    got = gpu_run(cs, a, b)
    im, jn = sample_indices(cs.M, cs.N, count)
    want = oracle_sampled(cs, a, b, im, jn)
    assert_bits_equal(got[im, jn], want, cs.name + " (sampled)")
    return got


# ---------------------------------------------------------------------------
# the five workloads
_INPUTS = {}


def inputs(cs):
    """The case's operands, drawn once per recipe (the variants of a workload share them)."""
    key = (cs.M, cs.N, cs.K, cs.fmt_a, cs.fmt_b, cs.gen, cs.seed, cs.sigma_a, cs.sigma_b)
    if key not in _INPUTS:
        _INPUTS[key] = W.make_inputs(cs)
    return _INPUTS[key]


def all_indices(M, N):
    im, jn = np.meshgrid(np.arange(M, dtype=np.int64), np.arange(N, dtype=np.int64), indexing="ij")
    return im.ravel(), jn.ravel()


def stripe_check(cs, got, a, b, rows, cols):
    """A full-size row stripe and column stripe of the output against the oracle."""
    import oracle
    kw = dict(scale_result=cs.scale_result)
    want = oracle.scaled_mm(a[rows], b, cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b, cs.out_dtype,
                            cs.fast_accum, cs.split_S, cs.preset, **kw)
    assert_bits_equal(got[rows], want, f"{cs.name} rows {rows.start}:{rows.stop}")
    want = oracle.scaled_mm(a, b[cols], cs.fmt_a, cs.fmt_b, cs.scale_a, cs.scale_b, cs.out_dtype,
                            cs.fast_accum, cs.split_S, cs.preset, **kw)
    assert_bits_equal(got[:, cols], want, f"{cs.name} cols {cols.start}:{cols.stop}")


def test_tiny_full():
    full_check(W.case("tiny"))


def test_linear_full():
    full_check(W.case("linear"))


@pytest.mark.parametrize("cs", W.CONFIGS["square"], ids=lambda c: c.name)
def test_square_ragged_full(cs):
    # several CTA tiles (64 x 32 for this slow shape) with ragged tails in M, N and K
    # (K % 128 = 16)
    full_check(W.shrink(cs, 200, 144, 1040))


@pytest.mark.parametrize("i,cs", list(enumerate(W.CONFIGS["square"])), ids=lambda x: getattr(x, "name", str(x)))
def test_square_full_size_stripes(i, cs):
    # 64 full rows and 64 full columns at offsets that straddle CTA tiles (about 1e9
    # MACs each for the oracle), plus sampled outputs anywhere
    a, b = inputs(cs)
    got = gpu_run(cs, a, b)
    r0, c0 = 1000 + 517 * i, 3000 - 389 * i
    stripe_check(cs, got, a, b, slice(r0, r0 + 64), slice(c0, c0 + 64))
    im, jn = sample_indices(cs.M, cs.N, 96, seed=i)
    assert_bits_equal(got[im, jn], oracle_sampled(cs, a, b, im, jn), cs.name + " (sampled)")


_SPLITK_ACC = {}


@pytest.mark.parametrize("cs", W.CONFIGS["splitk"], ids=lambda c: c.name)
def test_splitk_full_size_every_output(cs):
    # all 16 x 256 outputs at K = 262144: the oracle's accumulators are computed once
    # per (preset, S, accumulation) and go through the epilogue of each output dtype
    import oracle
    a, b = inputs(cs)
    got = gpu_run(cs, a, b)
    key = (cs.preset, cs.split_S, cs.fast_accum)
    if key not in _SPLITK_ACC:
        im, jn = all_indices(cs.M, cs.N)
        _SPLITK_ACC[key] = oracle.acc_sampled(a, b, cs.fmt_a, cs.fmt_b, im, jn, cs.fast_accum,
                                              cs.split_S, cs.preset)
    want = oracle.epilogue(_SPLITK_ACC[key], cs.scale_a, cs.scale_b, cs.out_dtype)
    assert_bits_equal(got, want.reshape(cs.M, cs.N), cs.name)


@pytest.mark.parametrize("cs", [c for c in W.CONFIGS["splitk"] if c.out_dtype == "f32"],
                         ids=lambda c: c.name)
def test_splitk_ragged_full(cs):
    # K not a multiple of the 128 (64) k-tile: the short tile is the last of its split
    full_check(W.shrink(cs, 16, 64, 16384 + 48))


@pytest.mark.parametrize("i,cs", list(enumerate(W.CONFIGS["projection"])), ids=lambda x: getattr(x, "name", str(x)))
def test_projection_full_size_stripes_and_ragged(i, cs):
    a, b = inputs(cs)
    got = gpu_run(cs, a, b)
    r0, c0 = 4100 - 37 * i, 1000 + 21 * i
    stripe_check(cs, got, a, b, slice(r0, r0 + 64), slice(c0, c0 + 64))
    im, jn = sample_indices(cs.M, cs.N, 128, seed=i)
    assert_bits_equal(got[im, jn], oracle_sampled(cs, a, b, im, jn), cs.name + " (sampled)")
    full_check(W.shrink(cs, 272, 208, 1920))


# the fp32 accumulator entry point ("User guide", section 3: both operands as
# [rows, K]; the accumulator before the scales): every output against the oracle's
# accumulator, NaN rows and columns included
@pytest.mark.parametrize("fast", (True, False))
@pytest.mark.parametrize("S,preset", ((1, "hopper"), (2, "hopper"), (3, "ada")))
def test_accumulate_is_the_oracle_accumulator(fast, S, preset):
    import oracle
    from bit_exact_fp8_gb300 import accumulate
    cs = W.Case("acc", 40, 96, 1040, out_dtype="f32", fast_accum=fast, split_S=S, preset=preset,
                gen="mixed", seed=13)
    a, b = W.make_inputs(cs)
    a[3, 77] = 0x7F                      # NaN code in row 3
    b[5, 500] = 0xFF                     # NaN code in column 5
    dev = torch.device("cuda:0")
    x = torch.from_numpy(a).to(dev).view(torch.float8_e4m3fn)
    w = torch.from_numpy(b).to(dev).view(torch.float8_e4m3fn)
    got = accumulate(x, w, fast, splitk=S, preset=preset)
    torch.cuda.synchronize()
    got = got.cpu().view(torch.int32).numpy().view(np.uint32)
    im, jn = all_indices(cs.M, cs.N)
    want = oracle.acc_sampled(a, b, cs.fmt_a, cs.fmt_b, im, jn, fast, S, preset).reshape(cs.M, cs.N)
    assert_bits_equal(got, want, f"accumulate fast={fast} S={S} {preset}")
    assert (got[3] == 0x7FC00000).all() and (got[:, 5] == 0x7FC00000).all()
    assert not (got == 0x80000000).any()          # the accumulator is never -0


# ---------------------------------------------------------------------------
# presets x accumulation x output dtypes x formats on a ragged mid-size shape
@pytest.mark.parametrize("preset", ("hopper", "ada"))
@pytest.mark.parametrize("fast", (True, False))
@pytest.mark.parametrize("od", ("f32", "bf16", "f16"))
@pytest.mark.parametrize("fa,fb", (("e4m3fn", "e4m3fn"), ("e4m3fn", "e5m2"), ("e5m2", "e4m3fn")))
def test_matrix(preset, fast, od, fa, fb):
    cs = W.Case(f"matrix-{preset}-{fast}-{od}-{fa}-{fb}", 70, 96, 528, fa, fb, od, fast_accum=fast,
                preset=preset, gen="mixed", seed=7)
    full_check(cs)


@pytest.mark.parametrize("S", (2, 3, 5, 8, 24, 64))
@pytest.mark.parametrize("preset", ("hopper", "ada"))
@pytest.mark.parametrize("pairwise", (False, True))
def test_split_factors_and_combine(S, preset, pairwise):
    if pairwise and preset == "hopper":
        pytest.skip("the hopper preset combines serially")
    P = dict(block_width=32, frac_bits=13, restart=128, c_in_alignment=1, split_scheme=0,
             ktile=128, combine=0) if preset == "hopper" else \
        dict(block_width=16, frac_bits=13, restart=128, c_in_alignment=1, split_scheme=1,
             ktile=64, combine=int(pairwise))
    for fast in (True, False):
        cs = W.Case(f"split-{preset}-S{S}-{pairwise}-{fast}", 20, 48, 64 * 37 + 32, out_dtype="f32",
                    fast_accum=fast, split_S=S, preset=preset, seed=9, sigma_a=8.0, sigma_b=8.0)
        a, b = W.make_inputs(cs)
        got = gpu_run(cs, a, b, preset=P)
        want = oracle_full(cs, a, b, preset=P)
        assert_bits_equal(got, want, cs.name)


# ---------------------------------------------------------------------------
# edge and degenerate cases
def test_zero_dims_and_k0():
    from bit_exact_fp8_gb300 import scaled_mm
    dev = torch.device("cuda:0")
    one = torch.ones((), dtype=torch.float32, device=dev)
    for M, N in ((0, 32), (8, 0)):
        x = torch.zeros(M, 32, device=dev).to(torch.float8_e4m3fn)
        w = torch.zeros(N, 32, device=dev).to(torch.float8_e4m3fn)
        y = scaled_mm(x, w.t(), one, one, out_dtype=torch.bfloat16, use_fast_accum=True)
        assert y.shape == (M, N)
    x = torch.zeros(5, 0, device=dev).to(torch.float8_e4m3fn)
    w = torch.zeros(16, 0, device=dev).to(torch.float8_e4m3fn)
    y = scaled_mm(x, w.t(), one, -one, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), torch.zeros(5, 16, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (1, 16, 32), (3, 16, 48), (129, 80, 160),
                                   (257, 16, 16), (5, 1024, 16)])
def test_small_and_odd_shapes(M, N, K):
    for fast in (True, False):
        cs = W.Case(f"odd-{M}x{N}x{K}-{fast}", M, N, K, out_dtype="f32", fast_accum=fast,
                    gen="mixed", seed=M + N + K)
        full_check(cs)


@pytest.mark.parametrize("fmt", ("e4m3fn", "e5m2"))
def test_nan_rows_and_columns(fmt):
    cs = W.Case("nan", 40, 48, 256, fmt, "e4m3fn", "f32", fast_accum=False, split_S=3, seed=2)
    a, b = W.make_inputs(cs)
    a[7, 100] = 0x7F if fmt == "e4m3fn" else 0x7E
    b[13, 255] = 0xFF
    got = gpu_run(cs, a, b)
    want = oracle_full(cs, a, b)
    assert_bits_equal(got, want, "nan")
    assert (got[7] == 0x7FC00000).all() and (got[:, 13] == 0x7FC00000).all()


def test_inf_codes_ieee_reading():
    cs = W.Case("inf", 24, 32, 192, "e5m2", "e4m3fn", "f32", fast_accum=True, seed=3)
    a, b = W.make_inputs(cs)
    a[2, 10] = 0x7C            # +Inf
    a[5, 11] = 0xFC            # -Inf
    a[5, 40] = 0x7C            # +Inf and -Inf in one row -> NaN
    b[:, 60] = 0x00
    a[9, 60] = 0x7C            # Inf * 0 -> NaN
    for od in ("f32", "bf16", "f16"):
        c2 = W.Case("inf", 24, 32, 192, "e5m2", "e4m3fn", od, fast_accum=True, seed=3)
        assert_bits_equal(gpu_run(c2, a, b), oracle_full(c2, a, b), f"inf {od}")


def test_independent_of_out_buffer_and_deterministic():
    cs = W.shrink(W.case("linear"), 64, 320, 1920)
    a, b = W.make_inputs(cs)
    want = oracle_full(cs, a, b)
    for fill in (0x00, 0xFF, 0x7F):
        assert_bits_equal(gpu_run(cs, a, b, prefill=fill), want, f"prefill {fill:#x}")


def test_scales_zero_sign_and_specials():
    cs = W.Case("scales", 32, 32, 128, out_dtype="f32", seed=4)
    a, b = W.make_inputs(cs)
    for sa, sb in ((1.0, -1.0), (0.0, 1.0), (-0.0, 1.0), (1e-30, 1e-20), (3.0, float("inf")),
                   (float("nan"), 1.0), (1e-45, 1.0)):
        for od in ("f32", "bf16", "f16"):
            c2 = W.Case("scales", 32, 32, 128, out_dtype=od, scale_a=sa, scale_b=sb, seed=4)
            assert_bits_equal(gpu_run(c2, a, b), oracle_full(c2, a, b), f"scales {sa} {sb} {od}")


def test_rejections():
    from bit_exact_fp8_gb300 import ReferenceRejectsError, UnsupportedFeatureError, scaled_mm
    dev = torch.device("cuda:0")
    one = torch.ones((), dtype=torch.float32, device=dev)
    x = torch.zeros(16, 32, device=dev).to(torch.float8_e5m2)
    w = torch.zeros(16, 32, device=dev).to(torch.float8_e5m2)
    bf = torch.bfloat16
    with pytest.raises(ReferenceRejectsError):
        scaled_mm(x, w.t(), one, one, out_dtype=bf)        # e5m2 x e5m2
    x4 = torch.zeros(16, 40, device=dev).to(torch.float8_e4m3fn)
    w4 = torch.zeros(16, 40, device=dev).to(torch.float8_e4m3fn)
    with pytest.raises(ReferenceRejectsError):
        scaled_mm(x4, w4.t(), one, one, out_dtype=bf)      # K % 16
    x4 = torch.zeros(16, 32, device=dev).to(torch.float8_e4m3fn)
    with pytest.raises(ReferenceRejectsError):
        scaled_mm(x4, torch.zeros(32, 16, device=dev).to(torch.float8_e4m3fn), one, one,
                  out_dtype=bf)                            # mat2 row-major [K, N]
    with pytest.raises(UnsupportedFeatureError):
        scaled_mm(x4, x4.t(), torch.ones(16, 1, device=dev), one, out_dtype=bf)  # row-wise
    with pytest.raises(UnsupportedFeatureError):
        scaled_mm(x4, x4.t(), one, one, out_dtype=bf, splitk=65)


# fp8 outputs: scale_result as a separate fp32 multiply, then saturating
# round-to-nearest-even conversion ("Validation evidence", claims table)
@pytest.mark.parametrize("od", ("e4m3fn", "e5m2"))
@pytest.mark.parametrize("sr", (None, 0.37, -3.0, 1e-6))
@pytest.mark.parametrize("fa,fb", (("e4m3fn", "e4m3fn"), ("e4m3fn", "e5m2"), ("e5m2", "e4m3fn")))
def test_fp8_outputs(od, sr, fa, fb):
    if fa == fb == "e4m3fn" and od == "e5m2":
        pytest.skip("rejected: e4m3 x e4m3 -> e5m2")
    for fast, S in ((True, 1), (False, 3)):
        cs = W.Case(f"fp8-{od}-{sr}-{fa}-{fb}-{S}", 70, 96, 528, fa, fb, od, fast_accum=fast,
                    split_S=S, gen="mixed", seed=11, scale_a=1.0, scale_b=0.25, scale_result=sr)
        full_check(cs)


def test_fp8_output_rejection_and_k0():
    from bit_exact_fp8_gb300 import ReferenceRejectsError, scaled_mm
    dev = torch.device("cuda:0")
    one = torch.ones((), dtype=torch.float32, device=dev)
    x = torch.zeros(16, 32, device=dev).to(torch.float8_e4m3fn)
    with pytest.raises(ReferenceRejectsError):
        scaled_mm(x, x.t(), one, one, out_dtype=torch.float8_e5m2)
    x0 = torch.zeros(5, 0, device=dev).to(torch.float8_e4m3fn)
    w0 = torch.zeros(16, 0, device=dev).to(torch.float8_e4m3fn)
    y = scaled_mm(x0, w0.t(), one, one, scale_result=-one, out_dtype=torch.float8_e4m3fn)
    torch.cuda.synchronize()
    # fma(+0, alpha, +0) = +0, times -1 = -0: code 0x80
    assert (y.view(torch.uint8) == 0x80).all()
