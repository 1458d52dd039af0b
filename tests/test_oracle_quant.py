"""Pins for the oracle's quantizer: values and properties the pages fix.

"O Seu Cache KV Nao Tem um Problema de Bits...", section "O Que o Erro de
Quantizacao E Realmente Feito": zero point = group minimum, step = range /
(2^B - 1), each element rounded to the nearest step, error at most half a
step, one outlier inflates the step of its whole group.  "Kuantisasi KV Cache
untuk Mengurangi Memory Inferensi Long Context", section "Scale menentukan
sistem koordinat kuantisasi": symmetric q = clamp(round(x/scale)), x_hat =
q*scale.  Sections "Chaves..." / "Valores..." of the first page fix the
grouping axes (keys along tokens per channel, values along channels per token).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def _ulp32(a):
    return np.spacing(np.abs(np.float32(a))).astype(np.float64)


def _check_group(x, bits, sym, meta_f32):
    x = np.asarray(x, np.float32)
    codes, z, s = oracle.quant_group(x, bits, sym, meta_f32)
    levels = (1 << bits) - 1
    xhat = np.array([oracle.dequant_one(int(c), z, s, bits, sym) for c in codes])
    slack = 8 * max(_ulp32(np.max(np.abs(x))), _ulp32(z))
    # codes in range
    if sym:
        qmax = (1 << (bits - 1)) - 1
        assert codes.min() >= (1 << (bits - 1)) - qmax and codes.max() <= (1 << (bits - 1)) + qmax
    else:
        assert codes.max() <= levels
    # half-step error bound
    err = np.abs(x.astype(np.float64) - xhat)
    assert np.all(err <= float(s) / 2 * (1 + 1e-6) + slack), (err.max(), s)
    # monotone
    order = np.argsort(x, kind="stable")
    assert np.all(np.diff(codes[order].astype(int)) >= 0)
    # nearest level in exact arithmetic, given the stored (z, s); near-ties may go either way
    if s != 0:
        S, Z = Fraction(float(s)), Fraction(float(z))
        off = (1 << (bits - 1)) if sym else 0
        lo = 1 if sym else 0
        for xi, ci in zip(x, codes):
            X = Fraction(float(xi))
            d = [abs(X - ((q - off) * S + (0 if sym else Z))) for q in range(lo, levels + 1)]
            best = min(d)
            mine = d[int(ci) - lo]
            assert mine - best <= Fraction(1, 10**6) * S + Fraction(float(slack)), (xi, ci)
    return codes, z, s


def test_tie_example_from_page():
    g = GOLD["tie_example"]
    codes, z, s = oracle.quant_group(g["group"], g["bits"])
    assert z == g["zero"] and s == g["step"]
    assert codes.tolist() == g["codes"]


def test_single_outlier_inflates_the_group():
    g = GOLD["outlier_example"]
    rng = np.random.default_rng(0)
    small = rng.uniform(*g["small_range"], size=g["n_small"]).astype(np.float32)
    x = np.concatenate([small, np.float32([g["outlier"]])])
    codes, z, s = _check_group(x, g["bits"], False, False)
    mn = float(np.float16(small.min()).astype(np.float32))
    # closed form: step = (outlier - min) / 3, stored rounded up to fp16
    assert abs(float(s) - (g["outlier"] - small.min()) / 3) < 0.05
    assert np.all(codes[:-1] == g["small_codes"]) and codes[-1] == 3
    assert mn >= -1.0
    # at 8 bits the 31 small values share at most 6 of the 256 codes
    codes8, _, s8 = _check_group(x, 8, False, False)
    assert len(set(codes8[:-1].tolist())) <= 6


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("meta_f32", [False, True])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("n", [2, 4, 32])
def test_random_groups_properties(bits, meta_f32, sym, n):
    rng = np.random.default_rng(bits * 100 + n + 7 * sym + 3 * meta_f32)
    for trial in range(6):
        scale = [1e-3, 1.0, 30.0][trial % 3]
        x = (rng.standard_normal(n) * scale).astype(np.float32)
        if trial >= 3:
            x = x.astype(np.float16).astype(np.float32)
        _check_group(x, bits, sym, meta_f32)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_metadata_rounding_directions(bits):
    rng = np.random.default_rng(bits)
    levels = (1 << bits) - 1
    for _ in range(200):
        x = (rng.standard_normal(32) * rng.uniform(0.01, 50)).astype(np.float32)
        _, z, s = oracle.quant_group(x, bits)
        zh = np.float16(z)
        assert np.float32(zh) == z  # stored as fp16
        # zero point = the largest fp16 not above the group minimum
        assert float(z) <= float(x.min()) < float(np.nextafter(zh, np.float16(np.inf)))
        # step = the smallest fp16 not below the fp32 quotient (max - z) / (2^B - 1)
        q32 = np.float32(np.float32(x.max() - z) / np.float32(levels))
        sh = np.float16(s)
        assert float(s) >= float(q32) > float(np.nextafter(sh, np.float16(-np.inf)))


def test_fp32_metadata_is_the_literal_formula():
    rng = np.random.default_rng(5)
    for bits in (2, 4, 8):
        x = rng.standard_normal(64).astype(np.float32)
        codes, z, s = oracle.quant_group(x, bits, meta_f32=True)
        assert z == x.min()
        assert s == np.float32(np.float32(x.max() - x.min()) / np.float32((1 << bits) - 1))
        assert codes[np.argmin(x)] == 0 and codes[np.argmax(x)] == (1 << bits) - 1


def test_symmetric_extremes_and_offset():
    x = np.array([-3.0, -1.0, 0.0, 0.25, 3.0], np.float32)
    for bits in (2, 4, 8):
        qmax = (1 << (bits - 1)) - 1
        codes, z, s = oracle.quant_group(x, bits, sym=True, meta_f32=True)
        assert z == 0 and s == np.float32(3.0) / np.float32(qmax)
        off = 1 << (bits - 1)
        assert codes[0] == off - qmax and codes[-1] == off + qmax and codes[2] == off
        for c, xi in zip(codes, x):
            assert oracle.dequant_one(int(c), z, s, bits, True) == pytest.approx(
                float(np.clip(np.rint(xi / s), -qmax, qmax)) * float(s))


def test_zero_range_and_negative_zero():
    codes, z, s = oracle.quant_group(np.full(32, 1.5, np.float32), 4)
    assert s == 0 and z == 1.5 and not codes.any()
    assert oracle.dequant_one(0, z, s, 4) == 1.5
    codes, z, s = oracle.quant_group(np.full(8, -0.0, np.float32), 3)
    assert np.float32(z).view(np.uint32) == 0 and np.float32(s).view(np.uint32) == 0
    codes, z, s = oracle.quant_group(np.full(8, -0.0, np.float32), 3, meta_f32=True)
    assert np.float32(z).view(np.uint32) == 0 and np.float32(s).view(np.uint32) == 0


# ----------------------------------------------------------- tensor level ---

def _tensor(batch=2, T=70, H=3, D=64, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, T, H, D)).astype(np.float16).astype(np.float32)
    return x


@pytest.mark.parametrize("axis,group", [(oracle.PER_CHANNEL, 32), (oracle.PER_TOKEN, 32),
                                        (oracle.PER_TOKEN, 64), (oracle.PER_TOKEN, oracle.WHOLE_VECTOR)])
def test_group_membership_locality(axis, group):
    """Changing one element changes only the metadata of its own group: this pins
    the grouping axis (a transposed group would move other groups)."""
    x = _tensor()
    lens = np.array([70, 45], np.int32)
    tcap = 96
    base = oracle.quantize_tensor(x, lens, tcap, 4, group, axis)
    b, t, h, c = 1, 20, 2, 17
    x2 = x.copy()
    x2[b, t, h, c] = 50.0
    pert = oracle.quantize_tensor(x2, lens, tcap, 4, group, axis)
    changed = np.nonzero(np.any(base["meta"] != pert["meta"], axis=1))[0].tolist()
    H, D = x.shape[2], x.shape[3]
    if axis == oracle.PER_CHANNEL:
        expect = [((b * H + h) * (tcap // group) + t // group) * D + c]
    elif group == oracle.WHOLE_VECTOR:
        expect = [b * tcap + t]
    else:
        expect = [((b * H + h) * tcap + t) * (D // group) + c // group]
    assert changed == expect


def test_per_channel_tail_and_sealed_counts():
    x = _tensor()
    lens = np.array([70, 45], np.int32)
    q = oracle.quantize_tensor(x, lens, 96, 3, 32, oracle.PER_CHANNEL)
    assert oracle.sealed(70, oracle.PER_CHANNEL, 32) == 64 and oracle.sealed(45, oracle.PER_CHANNEL, 32) == 32
    # tail = the unsealed tokens rounded to nearest fp16 (inputs here are fp16 already: identity)
    tail = q["tail"]
    np.testing.assert_array_equal(tail[0, :, :6, :], x[0, 64:70].transpose(1, 0, 2).astype(np.float16).view(np.uint16))
    np.testing.assert_array_equal(tail[1, :, :13, :], x[1, 32:45].transpose(1, 0, 2).astype(np.float16).view(np.uint16))
    # codes beyond the sealed tokens stay 0
    assert not q["codes"][0, :, 64:, :].any() and not q["codes"][1, :, 32:, :].any()
    xh = oracle.dequant_tensor(q, lens, 3, 32, oracle.PER_CHANNEL)
    np.testing.assert_array_equal(xh[0, :, 64:70, :], x[0, 64:70].transpose(1, 0, 2).astype(np.float64))


@pytest.mark.parametrize("axis,group", [(oracle.PER_CHANNEL, 32), (oracle.PER_CHANNEL, 64),
                                        (oracle.PER_TOKEN, 32), (oracle.PER_TOKEN, oracle.WHOLE_VECTOR)])
@pytest.mark.parametrize("bits", [2, 3, 6])
@pytest.mark.parametrize("sym", [False, True])
def test_tensor_error_bound(axis, group, bits, sym):
    x = _tensor(seed=bits)
    lens = np.array([70, 64], np.int32)
    tcap = 128
    q = oracle.quantize_tensor(x, lens, tcap, bits, group, axis, sym)
    xh = oracle.dequant_tensor(q, lens, bits, group, axis, sym)
    xt = x.transpose(0, 2, 1, 3)
    H, D = x.shape[2], x.shape[3]
    g = oracle.resolve_group(group, H, D)
    for b, n in enumerate(lens):
        ns = oracle.sealed(int(n), axis, g)
        err = np.abs(xh[b, :, :ns, :] - xt[b, :, :ns, :])
        # step of each element's group
        meta = q["meta"]
        step = np.empty_like(err)
        for h in range(H):
            for t in range(ns):
                for c in range(D):
                    if axis == oracle.PER_CHANNEL:
                        mi = ((b * H + h) * (tcap // g) + t // g) * D + c
                    elif g == H * D:
                        mi = b * tcap + t
                    else:
                        mi = ((b * H + h) * tcap + t) * (D // g) + c // g
                    step[h, t, c] = meta[mi, 1]
        assert np.all(err <= step / 2 * (1 + 1e-6) + 1e-6)


def test_outlier_channels_per_channel_keys_beat_per_token_keys():
    """Keys with a few fixed large channels: grouping along tokens per channel
    isolates them, grouping along channels per token spreads their range over
    every token's group, so per-channel reconstruction error is smaller."""
    rng = np.random.default_rng(0)
    B, T, H, D = 1, 256, 4, 64
    x = rng.standard_normal((B, T, H, D)).astype(np.float32)
    ordinary = np.ones((H, D), bool)
    for h in range(H):
        ch = rng.choice(D, 2, replace=False)
        x[:, :, h, ch] *= 20.0
        ordinary[h, ch] = False
    lens = np.array([T], np.int32)
    errs = {}
    for axis in (oracle.PER_CHANNEL, oracle.PER_TOKEN):
        q = oracle.quantize_tensor(x, lens, T, 2, 32, axis)
        xh = oracle.dequant_tensor(q, lens, 2, 32, axis)
        e2 = (xh - x.transpose(0, 2, 1, 3)) ** 2  # [B][H][T][D]
        errs[axis] = e2[0].transpose(0, 2, 1)[ordinary].mean()
    # the ordinary channels pay for the outliers only under per-token grouping
    assert errs[oracle.PER_CHANNEL] < 0.1 * errs[oracle.PER_TOKEN]


def test_per_channel_groups_use_the_fp16_staging_values():
    """Tokens of an unsealed per-channel group wait in the fp16 tail, so a
    sealed group is quantized from the fp16-rounded values; a prefix of a
    sequence seals exactly the groups the longer sequence seals."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((1, 96, 2, 64)) * 3).astype(np.float32)  # fp32 source values
    lens = np.array([96], np.int32)
    a = oracle.quantize_tensor(x, lens, 96, 4, 32, oracle.PER_CHANNEL)
    x16 = x.astype(np.float16).astype(np.float32)
    b = oracle.quantize_tensor(x16, lens, 96, 4, 32, oracle.PER_CHANNEL)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["meta"], b["meta"])
    pre = oracle.quantize_tensor(x, np.array([70], np.int32), 96, 4, 32, oracle.PER_CHANNEL)
    np.testing.assert_array_equal(pre["codes"][:, :, :64], a["codes"][:, :, :64])
    mp = pre["meta"].reshape(1, 2, 3, 64, 2)
    ma = a["meta"].reshape(1, 2, 3, 64, 2)
    np.testing.assert_array_equal(mp[:, :, :2], ma[:, :, :2])


# ---------------------------------------------------------------------------
# Full-precision recent window ("O Seu Cache KV Nao Tem um Problema de Bits...",
# section "O Imposto dos Sistemas e Por Que Nao E um Detalhe": the newest
# tokens, up to 128, stay in full precision; groups are quantized once enough
# tokens have accumulated).  Reading: per-channel groups seal once all their
# tokens are older than the newest R; per-token tensors quantize 16-token
# blocks once all of the block is older than the newest R; tokens quantized
# after a stay in the window are quantized from their fp16 values.

@pytest.mark.parametrize("n,axis,group,window,expect", [
    (100, oracle.PER_CHANNEL, 32, 64, 32), (96, oracle.PER_CHANNEL, 32, 64, 32), (95, oracle.PER_CHANNEL, 32, 64, 0),
    (100, oracle.PER_CHANNEL, 32, 0, 96), (100, oracle.PER_TOKEN, 32, 32, 64), (47, oracle.PER_TOKEN, 32, 32, 0),
    (48, oracle.PER_TOKEN, 32, 32, 16), (100, oracle.PER_TOKEN, 32, 0, 100), (10, oracle.PER_TOKEN, 32, 128, 0)])
def test_window_sealed_counts(n, axis, group, window, expect):
    assert oracle.sealed(n, axis, group, window) == expect
    assert oracle.tail_rows(axis, group, window) == (group + window if axis == oracle.PER_CHANNEL
                                                     else (window + 16 if window else 0))


def _fp16_round(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


@pytest.mark.parametrize("axis,group", [(oracle.PER_TOKEN, 32), (oracle.PER_TOKEN, oracle.WHOLE_VECTOR),
                                        (oracle.PER_CHANNEL, 32), (oracle.PER_CHANNEL, 16)])
@pytest.mark.parametrize("window", [16, 64])
def test_window_keeps_recent_tokens_in_fp16(axis, group, window):
    rng = np.random.default_rng(7)
    B, T, H, D = 2, 150, 2, 64
    x = rng.standard_normal((B, T, H, D)).astype(np.float32)
    lens = [150, 77]
    tcap = 160
    q = oracle.quantize_tensor(x, lens, tcap, 4, group, axis, window=window)
    q0 = oracle.quantize_tensor(_fp16_round(x), lens, tcap, 4, group, axis, window=0)
    g = oracle.resolve_group(group, H, D)
    xh = oracle.dequant_tensor(q, lens, 4, group, axis, window=window)
    xh0 = oracle.dequant_tensor(q0, lens, 4, group, axis, window=0)
    for b, n in enumerate(lens):
        ns = oracle.sealed(n, axis, g, window)
        assert n - ns >= (window if n >= window else n)  # at least the newest R tokens stay fp16
        # window rows: the input rounded to nearest fp16, row t - sealed
        rows = q["tail"][b, :, : n - ns].view(np.float16).astype(np.float32)
        np.testing.assert_array_equal(rows, _fp16_round(x[b, ns:n]).transpose(1, 0, 2))
        np.testing.assert_array_equal(xh[b, :, ns:n], _fp16_round(x[b, ns:n]).transpose(1, 0, 2).astype(np.float64))
        # no codes past the sealed prefix
        assert not q["codes"][b, :, ns:].any()
        # the sealed prefix is what quantizing the fp16 values without a window gives
        np.testing.assert_array_equal(q["codes"][b, :, :ns], q0["codes"][b, :, :ns])
        np.testing.assert_array_equal(xh[b, :, :ns], xh0[b, :, :ns])


@pytest.mark.parametrize("axis", [oracle.PER_TOKEN, oracle.PER_CHANNEL])
def test_window_sealed_prefix_never_changes_as_tokens_arrive(axis):
    """A token's codes, once sealed, are the same for every later length
    (the window slides; nothing already quantized is requantized)."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 200, 2, 64)).astype(np.float32)
    prev = None
    for n in range(60, 200, 7):
        q = oracle.quantize_tensor(x, [n], 208, 3, 32, axis, window=48)
        ns = oracle.sealed(n, axis, 32, 48)
        if prev is not None:
            pq, pns = prev
            np.testing.assert_array_equal(q["codes"][0, :, :pns], pq["codes"][0, :, :pns])
        prev = (q, ns)


def test_window_byte_terms():
    lens = [150, 77]
    p, m, t = oracle.tensor_bytes(2, 3, 64, lens, 2, 32, oracle.PER_TOKEN, window=32)
    ns = [oracle.sealed(n, oracle.PER_TOKEN, 32, 32) for n in lens]
    assert ns == [112, 32]
    assert t == sum(n - s for n, s in zip(lens, ns)) * 3 * 64 * 2
    assert p == sum(ns) * 3 * 64 * 2 / 8
    assert m == sum(ns) * 3 * (64 // 32) * 4
