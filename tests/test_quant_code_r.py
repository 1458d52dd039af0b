"""The fused append's code rule through the step's reciprocal (quant_code_r in
bit_quantized_kv_02_gb300/csrc/kvq_common.cuh) gives the same code as the plain
rule with an IEEE division (quant_code, which the oracle also follows).

numpy's float32 operations round to nearest like __frcp_rn / __fmul_rn /
__fsub_rn / __fdiv_rn, so both rules are emulated exactly here and compared on
random groups and on quotients placed at and around half-integers, across the
2^-12 cutoff below which the reciprocal rule defers to the division.  The
prefill kernels' form of the rule (quant_code_fast: rounding by adding and
removing 1.5 * 2^23, the same cutoff read from the same sums) is emulated and
compared the same way."""
import numpy as np

F = np.float32


def code_div(x, z, s, bits, sym):
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        if sym:
            qmax = F((1 << (bits - 1)) - 1)
            t = np.rint(x / s)
            return (np.clip(t, -qmax, qmax) + F(1 << (bits - 1))).astype(np.int64)
        t = np.rint((x - z) / s)
        return np.clip(t, F(0), F((1 << bits) - 1)).astype(np.int64)


def code_rcp(x, z, s, bits, sym):
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        num = x if sym else (x - z).astype(F)
        r = (F(1) / s).astype(F)
        q0 = (num * r).astype(F)
        aq = np.abs(q0)
        fr = (aq - np.floor(aq)).astype(F)
        fast = (aq <= F(512)) & (r >= F(2.0 ** -125)) & (np.abs(fr - F(0.5)) > F(2.0 ** -12))
        t = np.where(fast, np.rint(q0), np.rint(num / s))
        if sym:
            qmax = F((1 << (bits - 1)) - 1)
            return (np.clip(t, -qmax, qmax) + F(1 << (bits - 1))).astype(np.int64)
        return np.clip(t, F(0), F((1 << bits) - 1)).astype(np.int64)


def code_magic(x, z, s, bits, sym):
    """The prefill kernels' form of the same rule (quant_code_fast): the
    quotient through the step's reciprocal (0 for a zero step), rounded to the
    nearest integer (ties to even) by adding and removing 1.5 * 2^23 in
    float32, the distance to that integer from the same sums; near a
    half-integer, for a quotient beyond 512 or a subnormal reciprocal the IEEE
    division decides; the integer code is clamped like the division rule."""
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        M = F(12582912.0)
        num = x if sym else (x - z).astype(F)
        r = np.where(s > 0, (F(1) / s).astype(F), F(0)).astype(F)
        q0 = (num * r).astype(F)
        c = ((q0 + M).astype(F) - M).astype(F)
        e = (q0 - c).astype(F)
        fast = (np.abs(q0) <= F(512)) & (np.abs(e) < F(0.5 - 2.0 ** -12)) & ((r >= F(2.0 ** -125)) | (s == 0))
        t = np.where(fast, c, np.rint(num / s)).astype(np.float64)
        t = np.where(s == 0, 0.0, t)
        if sym:
            qmax = (1 << (bits - 1)) - 1
            return (np.clip(t, -qmax, qmax) + (1 << (bits - 1))).astype(np.int64)
        return np.clip(t, 0, (1 << bits) - 1).astype(np.int64)


def fp16_steps(rng, n, lo=-14, hi=8):
    """Positive steps as stored in fp16 metadata (normal fp16 values)."""
    return np.ldexp(1.0 + rng.integers(0, 1024, n) / 1024.0, rng.integers(lo, hi, n)).astype(F)


def test_random_groups_agree():
    rng = np.random.default_rng(0)
    for bits in (2, 3, 4, 5, 6, 7, 8):
        n = 400_000
        s = fp16_steps(rng, n)
        z = (rng.standard_normal(n) * 4).astype(np.float16).astype(F)
        levels = (1 << bits) - 1
        x = (z + rng.uniform(-0.1, levels + 0.1, n).astype(F) * s).astype(F)
        for sym in (False, True):
            np.testing.assert_array_equal(code_rcp(x, z, s, bits, sym), code_div(x, z, s, bits, sym))
            np.testing.assert_array_equal(code_magic(x, z, s, bits, sym), code_div(x, z, s, bits, sym))


def test_quotients_around_half_integers_agree():
    rng = np.random.default_rng(1)
    offsets = np.array([0.0, 2.0 ** -24, 2.0 ** -20, 2.0 ** -14, 2.0 ** -13, 2.0 ** -12 - 2.0 ** -18, 2.0 ** -12,
                        2.0 ** -12 + 2.0 ** -18, 2.0 ** -11, 2.0 ** -9, 1e-3])
    offsets = np.concatenate([offsets, -offsets])
    for bits in (2, 4, 8):
        levels = (1 << bits) - 1
        n = 200_000
        s = fp16_steps(rng, n)
        z = (rng.standard_normal(n) * 2).astype(np.float16).astype(F)
        k = rng.integers(0, levels, n)
        d = offsets[rng.integers(0, len(offsets), n)]
        x = (z.astype(np.float64) + (k + 0.5 + d) * s.astype(np.float64)).astype(F)
        np.testing.assert_array_equal(code_rcp(x, z, s, bits, False), code_div(x, z, s, bits, False))
        np.testing.assert_array_equal(code_magic(x, z, s, bits, False), code_div(x, z, s, bits, False))
        xs = ((rng.integers(0, 2, n) * 2 - 1) * (k + 0.5 + d) * s.astype(np.float64)).astype(F)
        np.testing.assert_array_equal(code_rcp(xs, z, s, bits, True), code_div(xs, z, s, bits, True))
        np.testing.assert_array_equal(code_magic(xs, z, s, bits, True), code_div(xs, z, s, bits, True))


def test_cutoff_takes_the_division_near_ties():
    # exact ties and quotients within the cutoff go through the division (half to even)
    s = np.full(4, F(0.1), dtype=F)
    z = np.zeros(4, dtype=F)
    x = (np.array([2.5, 3.5, 2.5 + 2.0 ** -14, 3.5 - 2.0 ** -14]) * np.float64(F(0.1))).astype(F)
    np.testing.assert_array_equal(code_rcp(x, z, s, 4, False), code_div(x, z, s, 4, False))
    np.testing.assert_array_equal(code_magic(x, z, s, 4, False), code_div(x, z, s, 4, False))


def test_degenerate_steps_agree():
    # zero, subnormal and huge steps, and NaN inputs, follow the division's outcome
    x = np.array([0.0, 1.0, -1.0, 3.0e38, np.nan, 1e-30], dtype=F)
    for s_val in (1e-40, 1e-30, 3.0e38, 1.0):
        s = np.full(x.shape, F(s_val), dtype=F)
        z = np.zeros(x.shape, dtype=F)
        for sym in (False, True):
            a = code_rcp(x, z, s, 4, sym)
            b = code_div(x, z, s, 4, sym)
            c = code_magic(x, z, s, 4, sym)
            ok = ~np.isnan(x)
            np.testing.assert_array_equal(a[ok], b[ok])
            np.testing.assert_array_equal(c[ok], b[ok])


def code_try_rows(x, z, s, bits, sym, row=8):
    """The prefill kernels' batched form (quant_code_try): every value through
    the reciprocal, the integer read from the float32 bits of q0 + 1.5 * 2^23
    (0x4B400000 + rint(q0) for |q0| < 2^22); a row of `row` consecutive values
    in which any value fails the test (quotient beyond 512 or within 2^-12 of a
    half-integer, or a subnormal reciprocal of a non-zero step) is recomputed
    whole with the division-checked rule."""
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        M = F(12582912.0)
        num = x if sym else (x - z).astype(F)
        r = np.where(s > 0, (F(1) / s).astype(F), F(0)).astype(F)
        q0 = (num * r).astype(F)
        m = (q0 + M).astype(F)
        e = (q0 - (m - M).astype(F)).astype(F)
        q = m.view(np.int32).astype(np.int64) - 0x4B400000
        ok = (np.abs(q0) <= F(512)) & (np.abs(e) < F(0.5 - 2.0 ** -12)) & ((r >= F(2.0 ** -125)) | (s == 0))
        if sym:
            qmax = (1 << (bits - 1)) - 1
            q = np.clip(q, -qmax, qmax) + (1 << (bits - 1))
        else:
            q = np.clip(q, 0, (1 << bits) - 1)
        row_ok = ok.reshape(-1, row).all(axis=1).repeat(row)
        return np.where(row_ok, q, code_magic(x, z, s, bits, sym))


def test_batched_rows_with_integer_bits_agree():
    """Random groups, quotients at and around half-integers, zero steps: the
    batched rule gives the division rule's code for every value, whether its
    row took the fast path or was recomputed."""
    rng = np.random.default_rng(5)
    offsets = np.array([0.0, 2.0 ** -24, 2.0 ** -13, 2.0 ** -12, 2.0 ** -11, 0.1, 0.37])
    offsets = np.concatenate([offsets, -offsets])
    for bits in (2, 3, 4, 6, 8):
        levels = (1 << bits) - 1
        n = 256_000
        s = fp16_steps(rng, n)
        s[rng.integers(0, n, 500)] = F(0)
        z = (rng.standard_normal(n) * 3).astype(np.float16).astype(F)
        k = rng.integers(0, levels, n)
        d = offsets[rng.integers(0, len(offsets), n)]
        x = (z.astype(np.float64) + (k + 0.5 + d) * s.astype(np.float64)).astype(F)
        for sym in (False, True):
            xx = x if not sym else ((rng.integers(0, 2, n) * 2 - 1) * (k + 0.5 + d) * s.astype(np.float64)).astype(F)
            got = code_try_rows(xx, z, s, bits, sym)
            # a zero step codes every value as 0 (the symmetric mid-code), as the oracle does
            want = np.where(s == 0, (1 << (bits - 1)) if sym else 0, code_div(xx, z, s, bits, sym))
            np.testing.assert_array_equal(got, want)
            assert (got >= 0).all() and (got <= levels).all()
