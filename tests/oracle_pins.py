"""Pins of the CPU oracle to facts fixed outside it.

Each ``pin_*`` function takes a loaded oracle library and raises
AssertionError if the oracle disagrees with something the pages or the
mathematics fix.  ``test_oracle_pins.py`` runs them on the oracle;
``test_oracle_mutants.py`` runs them on deliberately broken copies of it to
show that every plausible mistake is caught by at least one pin.

The sources of truth, none of which is the oracle itself:
  - numpy's binary16 <-> binary64 conversions (an independent codec),
  - exact integer arithmetic on the scaled fp16 values (``exact.py``),
  - numpy's float64 matmul within the textbook summation bound,
  - closed forms: all-ones products, the identity, zero padding,
  - the values "Quickstart: GPU" prints for its fill_42 and iota kernels,
    restated as products (``tests/golden``).
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle
from exact import F16_FORMAT, F32_FORMAT, distance_to_tie, exact_gemm_int48, round_rational

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U53 = Fraction(1, 2 ** 53)


def read_golden(name: str) -> np.ndarray:
    shape = None
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("shape:"):
                shape = tuple(int(s) for s in line.split(":")[1].split(","))
                continue
            vals.append(float(line))
    arr = np.array(vals, np.float64)
    assert shape is not None and arr.size == int(np.prod(shape)), name
    return arr.reshape(shape)


def _rand_f16(rng, shape, kind):
    """fp16 bit patterns with a chosen spread of exponents."""
    if kind == "uniform":
        x = rng.uniform(-1.0, 1.0, shape)
    elif kind == "wide":
        # magnitudes 2^-20 .. 2^4: normals and subnormals, both signs
        x = rng.choice([-1.0, 1.0], shape) * np.exp2(rng.uniform(-20.0, 4.0, shape))
    elif kind == "normal":
        x = rng.standard_normal(shape)
    else:
        raise ValueError(kind)
    return x.astype(np.float16).view(np.uint16)


# ---- the binary16 codec ------------------------------------------------------


def pin_decode_all_patterns(lib):
    """All 65 536 binary16 patterns decode exactly as numpy decodes them."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_f16(bits, lib=lib)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan), "NaN classification differs"
    assert np.array_equal(ours[~nan].view(np.uint64), ref[~nan].view(np.uint64)), \
        "decode differs from numpy on some finite/inf pattern"


def _f16_midpoints():
    """Every exact midpoint between neighbouring finite binary16 values, and
    the doubles just either side of it."""
    pos = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2.0  # exact in binary64
    mids = np.concatenate([mids, [65520.0]])  # the midpoint to the first overflow
    up = np.nextafter(mids, np.inf)
    dn = np.nextafter(mids, -np.inf)
    allv = np.concatenate([mids, up, dn])
    return np.concatenate([allv, -allv])


def pin_round_f16(lib):
    """binary64 -> binary16 rounding agrees bit for bit with numpy's direct
    conversion on every tie, both sides of every tie, random doubles over the
    whole range, subnormals, overflow and specials."""
    rng = np.random.default_rng(1234)
    rand = rng.choice([-1.0, 1.0], 1_000_000) * np.exp2(rng.uniform(-30.0, 17.0, 1_000_000))
    special = np.array([0.0, -0.0, 65504.0, 65519.999, 65520.0, 65536.0, 1e300, -1e300,
                        2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 2.0 ** -14,
                        2.0 ** -14 - 2.0 ** -25, 5e-324, np.inf, -np.inf])
    x = np.concatenate([_f16_midpoints(), rand, special])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    ours = oracle.round_f16(x, lib=lib)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} roundings differ, first x={x[bad[0]]!r}"
    nan_bits = oracle.round_f16(np.array([np.nan]), lib=lib)
    assert np.isnan(nan_bits.view(np.float16)).all()


def pin_round_f32(lib):
    """binary64 -> binary32 rounding agrees with numpy, through the product path."""
    rng = np.random.default_rng(99)
    # One-element products 1 x b reproduce b; then scale by a power of two so
    # the binary32 rounding of arbitrary doubles can be reached: use K=2 sums
    # a0*b0 + a1*b1 with values whose exact sum needs more than 24 bits.
    a = rng.uniform(-1, 1, (256, 2)).astype(np.float16)
    b = rng.uniform(-1, 1, (2, 256)).astype(np.float16)
    c64 = oracle.gemm(a, b, oracle.OUT_F64, lib=lib)
    c32 = oracle.gemm(a, b, oracle.OUT_F32, lib=lib)
    assert np.array_equal(c32.view(np.uint32), c64.astype(np.float32).view(np.uint32))
    for v in [1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, -(1.0 + 2.0 ** -24) , 2.0 ** -130]:
        assert np.float32(lib.oracle_f32_round(v)) == np.float32(np.float64(v))


# ---- the product ---------------------------------------------------------------


def _check_exact(lib, a_bits, b_bits):
    M, K = a_bits.shape
    N = b_bits.shape[1]
    exact = exact_gemm_int48(a_bits, b_bits)
    absprod = exact_gemm_int48(a_bits & 0x7FFF, b_bits & 0x7FFF)  # sum |a||b|, scaled
    c64 = oracle.gemm(a_bits, b_bits, oracle.OUT_F64, lib=lib)
    c16 = oracle.gemm(a_bits, b_bits, oracle.OUT_F16, lib=lib)
    c32 = oracle.gemm(a_bits, b_bits, oracle.OUT_F32, lib=lib)
    scale = Fraction(1, 2 ** 48)
    for i in range(M):
        for j in range(N):
            q = exact[i, j] * scale
            bound = K * U53 * absprod[i, j] * scale  # |fl(sum) - sum| <= K u sum|ab|
            got = Fraction(float(c64[i, j]))
            assert abs(got - q) <= bound, f"fp64 sum off at ({i},{j}): {float(got)} vs {float(q)}"
            for out, fmt, kind in ((c16, F16_FORMAT, "f16"), (c32, F32_FORMAT, "f32")):
                want = round_rational(q, fmt)
                if kind == "f16":
                    val = np.array([out[i, j]], np.uint16).view(np.float16)[0]
                else:
                    val = out[i, j]
                val = float(val)
                if isinstance(want, float):
                    ok = val == want
                else:
                    ok = np.isfinite(val) and Fraction(val) == want
                if not ok:
                    # only acceptable when the fp64 sum could sit on the other side of a tie
                    assert distance_to_tie(q, fmt) <= bound, \
                        f"{kind} rounding off at ({i},{j}): {val} vs {float(want)}"


def pin_exact_small(lib):
    """Brute force in exact integer arithmetic on products up to 64^3."""
    rng = np.random.default_rng(7)
    cases = [((1, 1, 1), "uniform"), ((3, 7, 5), "wide"), ((17, 9, 33), "uniform"),
             ((5, 40, 24), "normal"), ((64, 64, 64), "uniform"), ((13, 31, 64), "wide")]
    for (M, N, K), kind in cases:
        a = _rand_f16(rng, (M, K), kind)
        b = _rand_f16(rng, (K, N), kind)
        _check_exact(lib, a, b)


def pin_numpy_f64(lib):
    """Against numpy's float64 matmul of numpy-decoded inputs, within twice
    the textbook bound K u sum|a||b| (each side within one bound of exact)."""
    rng = np.random.default_rng(11)
    for (M, N, K), kind in [((96, 80, 200), "normal"), ((33, 130, 257), "wide"), ((8, 300, 64), "uniform")]:
        a = _rand_f16(rng, (M, K), kind)
        b = _rand_f16(rng, (K, N), kind)
        a64 = a.view(np.float16).astype(np.float64)
        b64 = b.view(np.float16).astype(np.float64)
        ref = a64 @ b64
        bound = 2.0 * K * 2.0 ** -53 * (np.abs(a64) @ np.abs(b64)) + 1e-300
        got = oracle.gemm(a, b, oracle.OUT_F64, lib=lib)
        assert np.all(np.abs(got - ref) <= bound), "fp64 sums differ from numpy matmul"


def pin_all_ones(lib):
    """All-ones A [M,K] and B [K,N] give C = K exactly (K a power of two is
    exact in binary16 and binary32)."""
    for K in (1, 64, 256, 4096, 8192, 32768):
        a = np.ones((3, K), np.float16)
        b = np.ones((K, 5), np.float16)
        c16 = oracle.gemm(a, b, oracle.OUT_F16, lib=lib).view(np.float16)
        c32 = oracle.gemm(a, b, oracle.OUT_F32, lib=lib)
        assert np.all(c16 == np.float16(K)), K
        assert np.all(c32 == np.float32(K)), K
    # 2049 is not a binary16 value: 2049 = 2048 + 1 ties to the even 2048
    a = np.ones((2, 2049), np.float16)
    b = np.ones((2049, 3), np.float16)
    assert np.all(oracle.gemm(a, b, oracle.OUT_F16, lib=lib).view(np.float16) == np.float16(2048))
    assert np.all(oracle.gemm(a, b, oracle.OUT_F32, lib=lib) == np.float32(2049))


def pin_identity(lib):
    """B = I returns A: bit for bit except that -0 sums to +0."""
    rng = np.random.default_rng(5)
    for M, K, kind in [(40, 72, "wide"), (7, 128, "normal")]:
        a = _rand_f16(rng, (M, K), kind)
        eye = np.eye(K, dtype=np.float16)
        c16 = oracle.gemm(a, eye, oracle.OUT_F16, lib=lib)
        c32 = oracle.gemm(a, eye, oracle.OUT_F32, lib=lib)
        a_clean = np.where(a == 0x8000, np.uint16(0), a)
        assert np.array_equal(c16, a_clean)
        assert np.array_equal(c32, a.view(np.float16).astype(np.float32))
        # A @ B with A = I returns B (checks the other operand's indexing)
        b = _rand_f16(rng, (K, M + 3), kind)
        c = oracle.gemm(np.eye(K, dtype=np.float16), b, oracle.OUT_F16, lib=lib)
        assert np.array_equal(c, np.where(b == 0x8000, np.uint16(0), b))


def pin_zero_padding(lib):
    """Zero columns of A against zero rows of B change nothing; zero rows of
    A and zero columns of B give zero rows and columns of C."""
    rng = np.random.default_rng(3)
    a = _rand_f16(rng, (30, 50), "normal")
    b = _rand_f16(rng, (50, 20), "normal")
    c = oracle.gemm(a, b, oracle.OUT_F16, lib=lib)
    ak = np.zeros((30, 64), np.uint16)
    ak[:, :50] = a
    bk = np.zeros((64, 20), np.uint16)
    bk[:50] = b
    assert np.array_equal(oracle.gemm(ak, bk, oracle.OUT_F16, lib=lib), c)
    am = np.zeros((37, 50), np.uint16)
    am[:30] = a
    bn = np.zeros((50, 29), np.uint16)
    bn[:, :20] = b
    cmn = oracle.gemm(am, bn, oracle.OUT_F16, lib=lib)
    assert np.array_equal(cmn[:30, :20], c)
    assert not cmn[30:].any() and not cmn[:, 20:].any()


def pin_fill_42(lib):
    """fill_42 as a product: ones[1,64] @ full[64,128] of 42/64 = 0.65625
    (exact in binary16) is 128 values of 42.0, as the quickstart prints."""
    want = read_golden("fill_42.txt")
    a = np.ones((1, 64), np.float16)
    b = np.full((64, 128), 0.65625, np.float16)
    for dt in (oracle.OUT_F16, oracle.OUT_F32):
        c = oracle.as_values(oracle.gemm(a, b, dt, lib=lib), dt).reshape(-1)
        assert np.array_equal(c, want)


def pin_iota(lib):
    """iota as a product: row i of A is [1, i] and B = [[0..127], [128]*128],
    so C[i, j] = j + 128 i, which flattened is 0..1023 as the quickstart
    prints for grid=(8,) blocks of 128."""
    want = read_golden("iota.txt")
    a = np.stack([np.ones(8), np.arange(8)], axis=1).astype(np.float16)
    b = np.stack([np.arange(128), np.full(128, 128)], axis=0).astype(np.float16)
    for dt in (oracle.OUT_F16, oracle.OUT_F32):
        c = oracle.as_values(oracle.gemm(a, b, dt, lib=lib), dt).reshape(-1)
        assert np.array_equal(c, want)


def pin_elems_and_threads(lib):
    """Element-wise entry point equals the row entry point, and results do not
    depend on the thread count or on which rows are asked for."""
    rng = np.random.default_rng(21)
    a = _rand_f16(rng, (37, 150), "normal")
    b = _rand_f16(rng, (150, 45), "normal")
    full1 = oracle.gemm(a, b, oracle.OUT_F64, nthreads=1, lib=lib)
    full7 = oracle.gemm(a, b, oracle.OUT_F64, nthreads=7, lib=lib)
    assert np.array_equal(full1.view(np.uint64), full7.view(np.uint64))
    rows = np.array([36, 0, 17, 17])
    part = oracle.gemm(a, b, oracle.OUT_F64, rows=rows, nthreads=3, lib=lib)
    assert np.array_equal(part.view(np.uint64), full1[rows].view(np.uint64))
    ii = rng.integers(0, 37, 200)
    jj = rng.integers(0, 45, 200)
    for dt in (oracle.OUT_F16, oracle.OUT_F32, oracle.OUT_F64):
        e = oracle.gemm_elems(a, b, ii, jj, dt, lib=lib)
        r = oracle.gemm(a, b, dt, lib=lib)[ii, jj]
        assert np.array_equal(e.view(np.uint8), r.view(np.uint8))


# ---- accumulation into an existing output ---------------------------------------


def pin_acc_zero_start_and_zero_product(lib):
    """Starting from zero is the plain product (bit for bit); a zero product
    returns the starting values (fp16 in, fp16 out: the same bits, with
    -0 + 0 = +0 as IEEE addition gives)."""
    rng = np.random.default_rng(31)
    a = _rand_f16(rng, (29, 70), "normal")
    b = _rand_f16(rng, (70, 41), "normal")
    zero16 = np.zeros((29, 41), np.uint16)
    for dt in (oracle.OUT_F16, oracle.OUT_F32, oracle.OUT_F64):
        assert np.array_equal(oracle.gemm_acc(a, b, zero16, dt, lib=lib).view(np.uint8),
                              oracle.gemm(a, b, dt, lib=lib).view(np.uint8))
    cin = _rand_f16(rng, (29, 41), "wide")
    got = oracle.gemm_acc(np.zeros((29, 70), np.uint16), b, cin, oracle.OUT_F16, lib=lib)
    assert np.array_equal(got, np.where(cin == 0x8000, np.uint16(0), cin))
    cin32 = rng.standard_normal((29, 41)).astype(np.float32)
    got32 = oracle.gemm_acc(np.zeros((29, 70), np.uint16), b, cin32, oracle.OUT_F32, lib=lib)
    assert np.array_equal(got32, cin32 + np.float32(0))


def pin_acc_all_ones(lib):
    """All-ones A and B from C = 3 give K + 3 exactly."""
    for K in (64, 4096):
        cin = np.full((3, 5), 3.0, np.float16)
        c = oracle.gemm_acc(np.ones((3, K), np.float16), np.ones((K, 5), np.float16), cin, oracle.OUT_F32,
                            lib=lib)
        assert np.all(c == np.float32(K + 3))


def pin_acc_exact(lib):
    """Exact integer brute force with a starting value, on a subset of rows in
    a scrambled order (so the starting value must be read from the source row,
    not the output position)."""
    rng = np.random.default_rng(41)
    for (M, N, K), kind in [((9, 13, 21), "wide"), ((16, 24, 48), "uniform")]:
        a = _rand_f16(rng, (M, K), kind)
        b = _rand_f16(rng, (K, N), kind)
        cin = _rand_f16(rng, (M, N), kind)
        exact = exact_gemm_int48(a, b)
        absprod = exact_gemm_int48(a & 0x7FFF, b & 0x7FFF)
        from exact import f16_to_int24
        cin48 = f16_to_int24(cin) * (1 << 24)
        rows = np.array([M - 1, 0, M // 2, 1])
        c64 = oracle.gemm_acc(a, b, cin, oracle.OUT_F64, rows=rows, lib=lib)
        c16 = oracle.gemm_acc(a, b, cin, oracle.OUT_F16, rows=rows, lib=lib)
        scale = Fraction(1, 2 ** 48)
        for r, i in enumerate(rows):
            for j in range(N):
                q = (exact[i, j] + cin48[i, j]) * scale
                bound = (K + 1) * U53 * (absprod[i, j] + abs(cin48[i, j])) * scale
                assert abs(Fraction(float(c64[r, j])) - q) <= bound
                want = round_rational(q, F16_FORMAT)
                val = float(np.array([c16[r, j]], np.uint16).view(np.float16)[0])
                ok = (val == want) if isinstance(want, float) else (np.isfinite(val) and Fraction(val) == want)
                if not ok:
                    assert distance_to_tie(q, F16_FORMAT) <= bound


def pin_acc_fp32_start(lib):
    """fp32 starting values: within the textbook bound of numpy's fp64
    Cin + A @ B."""
    rng = np.random.default_rng(43)
    a = _rand_f16(rng, (40, 90), "normal")
    b = _rand_f16(rng, (90, 33), "normal")
    cin = (rng.standard_normal((40, 33)) * 10).astype(np.float32)
    a64 = a.view(np.float16).astype(np.float64)
    b64 = b.view(np.float16).astype(np.float64)
    ref = cin.astype(np.float64) + a64 @ b64
    bound = 2.0 * 91 * 2.0 ** -53 * (np.abs(cin.astype(np.float64)) + np.abs(a64) @ np.abs(b64)) + 1e-300
    got = oracle.gemm_acc(a, b, cin, oracle.OUT_F64, lib=lib)
    assert np.all(np.abs(got - ref) <= bound)


# ---- the blocked add ----------------------------------------------------------


def pin_add_ieee_cases(lib):
    """Binary32 addition facts IEEE 754 fixes: exact small-integer sums, ties
    to even, signed zeros, subnormals, overflow to inf, inf - inf = NaN."""
    f = np.float32
    cases = [  # (x, y, x + y)
        (1.0, 2.0, 3.0),
        (1.0, 2.0 ** -24, 1.0),                      # halfway below 1 + ulp: ties to the even 1
        (1.0, 3 * 2.0 ** -24, 1.0 + 2.0 ** -22),     # halfway above: ties to even
        (-0.0, -0.0, -0.0), (-0.0, 0.0, 0.0), (5.0, -5.0, 0.0),
        (2.0 ** -149, 2.0 ** -149, 2.0 ** -148),      # subnormals add exactly
        (2.0 ** -126, -(2.0 ** -149), 2.0 ** -126 - 2.0 ** -149),
        (3.4028234663852886e38, 3.4028234663852886e38, np.inf),
        (np.inf, 1.0, np.inf),
    ]
    x = np.array([c[0] for c in cases], f)
    y = np.array([c[1] for c in cases], f)
    want = np.array([c[2] for c in cases], f)
    got = oracle.add_f32(x, y, lib=lib)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (got, want)
    assert np.isnan(oracle.add_f32(np.array([np.inf], f), np.array([-np.inf], f), lib=lib)).all()


def pin_add_against_numpy(lib):
    """Random binary32 operands over the whole exponent range, bit for bit
    against numpy's float32 addition (another IEEE implementation), and the
    pages' own check on their inputs' distribution: uniform [0, 1)."""
    rng = np.random.default_rng(61)
    x = (rng.choice([-1.0, 1.0], 200000) * np.exp2(rng.uniform(-140, 120, 200000))).astype(np.float32)
    y = (rng.choice([-1.0, 1.0], 200000) * np.exp2(rng.uniform(-140, 120, 200000))).astype(np.float32)
    assert np.array_equal(oracle.add_f32(x, y, lib=lib).view(np.uint32), (x + y).view(np.uint32))
    u = rng.random((512, 512), dtype=np.float32)
    v = rng.random((512, 512), dtype=np.float32)
    assert np.array_equal(oracle.add_f32(u, v, lib=lib), u + v)


ALL_PINS = [
    pin_decode_all_patterns,
    pin_round_f16,
    pin_round_f32,
    pin_exact_small,
    pin_numpy_f64,
    pin_all_ones,
    pin_identity,
    pin_zero_padding,
    pin_fill_42,
    pin_iota,
    pin_elems_and_threads,
    pin_acc_zero_start_and_zero_product,
    pin_acc_all_ones,
    pin_acc_exact,
    pin_acc_fp32_start,
    pin_add_ieee_cases,
    pin_add_against_numpy,
]
