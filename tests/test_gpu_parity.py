"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: codes, stored zero points / steps and fp16 tails bit-exact; decode
attention within 1e-3 of the oracle's fp64 attention over the same
dequantized cache, measured per (sequence, query head) as
max|out - ref| / max|ref|.  The 1e-3 bound is the path's stated tolerance; the
GPU computes in fp32 with ~22-bit operands, so typical errors are ~1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_02_gb300 import build, kvq, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


def make_cache(wl, max_tokens=None, max_splits=0, meta_dtype=kvq.F16, window=0):
    cfg = kvq.make_config(wl.layers, wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, max_tokens or wl.max_tokens,
                          wl.k, wl.v, meta_dtype, max_splits, window)
    return kvq.KVQCache(cfg)


def oracle_tensor(x_btHD, lens, tcap, tc, meta_f32, window=0):
    bits, group, axis, mode = tc
    return oracle.quantize_tensor(x_btHD.float().numpy(), np.array(lens, np.int32), tcap, bits, group, axis,
                                  bool(mode), bool(meta_f32), window)


def assert_export_equal(exp, orq, tc, which):
    codes = exp[f"codes_{which}"].cpu().numpy()
    meta = exp[f"meta_{which}"].cpu().numpy()
    np.testing.assert_array_equal(codes, orq["codes"], err_msg=f"codes_{which}")
    np.testing.assert_array_equal(meta.view(np.uint32), orq["meta"].view(np.uint32), err_msg=f"meta_{which}")
    if orq["tail"] is not None:
        tail = exp[f"tail_{which}"].cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(tail, orq["tail"], err_msg=f"tail_{which}")


def rel_err_rows(out, ref):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(out - ref).max(axis=-1)
    r = np.abs(ref).max(axis=-1)
    return d / np.maximum(r, 1e-30)


def decode_ref(wl, orq_k, orq_v, lens, q_cpu, scale, window=0):
    kh = oracle.dequant_tensor(orq_k, lens, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]), window)
    vh = oracle.dequant_tensor(orq_v, lens, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]), window)
    return oracle.attention(kh, vh, q_cpu.float().numpy(), np.array(lens, np.int32), scale)


def run_case(wl, lens, meta_f32=False, check_decode=True, layer=0, max_splits=0, generic=None, global_combine=False,
             window=0):
    """Prefill `lens` tokens of layer `layer`, compare the export and the decode output.
    generic: None keeps the default kernel choice, True forces the generic kernel,
    False requires the compile-time specialisation.  global_combine: merge the
    split-K partials through the global workspace even when a cluster could."""
    T = max(max(lens), 1)
    cache = make_cache(wl, max_tokens=T, max_splits=max_splits, meta_dtype=kvq.F32 if meta_f32 else kvq.F16,
                       window=window)
    if generic is True or global_combine:
        cache.kvq_set_decode_kernel((1 if generic else 0) | (2 if global_combine else 0))
    if generic is True:
        assert not cache.kvq_decode_kernel_specialized()
    elif generic is False:
        assert cache.kvq_decode_kernel_specialized()
    k, v = wl.layer_kv(layer, "cpu", T=T)
    lens_l = [int(x) for x in lens]
    cache.kvq_prefill_quantize(layer, k.cuda(), v.cuda(), lens_l)
    exp = cache.kvq_export(layer)
    torch.cuda.synchronize()
    ok = oracle_tensor(k, lens_l, cache.tcap, wl.k, meta_f32, window)
    ov = oracle_tensor(v, lens_l, cache.tcap, wl.v, meta_f32, window)
    assert_export_equal(exp, ok, wl.k, "k")
    assert_export_equal(exp, ov, wl.v, "v")
    assert exp["lens"].cpu().tolist() == lens_l
    if check_decode:
        q = wl.layer_query(layer)
        scale = np.float32(1.0 / np.sqrt(wl.head_dim))
        out = cache.kvq_decode_attn(layer, q.cuda(), scale=float(scale))
        torch.cuda.synchronize()
        assert cache.kvq_device_status() == 0
        ref = decode_ref(wl, ok, ov, lens_l, q, scale, window)
        err = rel_err_rows(out.cpu().numpy(), ref)
        for b, n in enumerate(lens_l):
            if n == 0:
                assert not out[b].any()
        assert err.max() <= TOL, (err.max(), np.unravel_index(err.argmax(), err.shape))
    return cache


def W(name, B, Hq, H, D, k, v, dtype=torch.float16, **kw):
    return synth.Workload(name, 1, B, Hq, H, D, [1], k, v, dtype, **kw)


PT, PC, ASYM, SYM, WHOLE = kvq.PER_TOKEN, kvq.PER_CHANNEL, kvq.ASYM, kvq.SYM, kvq.WHOLE_VECTOR


def test_tiny_config_parity():
    wl = synth.tiny()
    run_case(wl, wl.lens)


CASES = [
    # name, B, Hq, H, D, k cfg, v cfg, lens
    ("mha64_k4pc_v4pt", 2, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), [300, 77]),
    ("mha64_k2pc_v2pt_g64", 2, 3, 3, 64, (2, 64, PC, ASYM), (2, 64, PT, ASYM), [257, 64]),
    ("mha64_k3_v3", 1, 2, 2, 64, (3, 32, PC, ASYM), (3, 32, PT, ASYM), [200]),
    ("mha64_k5_v7", 1, 2, 2, 64, (5, 16, PC, ASYM), (7, 32, PT, ASYM), [129]),
    ("mha64_k6_v4_pt", 2, 2, 2, 64, (6, 64, PT, ASYM), (4, 64, PT, ASYM), [96, 33]),
    ("mha64_k8_v8", 1, 2, 2, 64, (8, 128, PC, ASYM), (8, 64, PT, ASYM), [390]),
    ("mha64_whole", 2, 4, 4, 64, (3, WHOLE, PT, ASYM), (3, WHOLE, PT, ASYM), [65, 140]),
    ("mha128_kt_vc", 2, 2, 2, 128, (2, 32, PT, ASYM), (2, 32, PC, ASYM), [113, 200]),
    ("mha128_kc_vc", 1, 3, 3, 128, (2, 32, PC, ASYM), (2, 32, PC, ASYM), [4096 + 17]),
    ("mha128_kt_vt", 1, 2, 2, 128, (2, 32, PT, ASYM), (2, 32, PT, ASYM), [161]),
    ("gqa2_128", 2, 4, 2, 128, (4, 64, PC, ASYM), (4, 64, PT, ASYM), [500, 1]),
    ("gqa4_128", 3, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), [1000, 64, 0]),
    ("gqa8_256_pt", 1, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [700]),
    ("gqa8_256_pc", 1, 16, 2, 256, (4, 32, PC, ASYM), (8, 32, PT, ASYM), [650]),
    ("gqa8_256_sym6", 1, 8, 1, 256, (6, 32, PT, SYM), (6, 32, PT, SYM), [333]),
    ("gqa8_256_vc", 1, 8, 1, 256, (3, 64, PC, SYM), (5, 64, PC, ASYM), [300]),
    ("sym_mha64", 2, 2, 2, 64, (4, 32, PC, SYM), (2, 32, PT, SYM), [150, 31]),
    # two queries x four value groups, one query x eight value groups (a step-scaled P operand per group)
    ("gqa2_128_vg4", 2, 4, 2, 128, (4, 32, PC, ASYM), (4, 32, PT, ASYM), [700, 50]),
    ("mha256_vg8", 2, 2, 2, 256, (4, 32, PT, ASYM), (5, 32, PT, ASYM), [500, 17]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_cases(case):
    name, B, Hq, H, D, kc, vc, lens = case
    wl = W(name, B, Hq, H, D, kc, vc, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=3)
    run_case(wl, lens)


# formats that have a compile-time specialisation of the decode kernel
FAST_CASES = [
    ("fast_d64_k4pc_v4pt", 2, 2, 2, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), [700, 65]),
    ("fast_d64_k6v4_pt64", 2, 2, 2, 64, (6, 64, PT, ASYM), (4, 64, PT, ASYM), [300, 17]),
    ("fast_d128_k2pc_v2pt", 2, 2, 2, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), [4113, 100]),
    ("fast_d128_gqa4", 2, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), [1500, 64]),
    ("fast_d256_gqa8_pt", 1, 8, 1, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [1000]),
    ("fast_d256_gqa8_pc", 1, 8, 1, 256, (4, 32, PC, ASYM), (8, 32, PT, ASYM), [777]),
    ("fast_d256_sym6", 1, 16, 2, 256, (6, 32, PT, SYM), (6, 32, PT, SYM), [600]),
    ("fast_d256_sym6_pc", 1, 16, 2, 256, (6, 32, PC, SYM), (6, 32, PT, SYM), [900]),
    ("fast_d256_gqa8_pt_ragged", 3, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [2049, 15, 0]),
]


@pytest.mark.parametrize("max_splits", [0, 2], ids=["planned", "two_splits"])
@pytest.mark.parametrize("kaxis", [PT, PC], ids=["kt", "kc"])
def test_d256_gqa8_global_merge(kaxis, max_splits):
    """The head_dim 256 specialisations with eight queries per kv head (keys
    per token and per channel) over a long and a short sequence: split-K
    partials merged through the global workspace, and with long warp ranges
    (two splits)."""
    wl = W("d256_pairs", 2, 16, 2, 256, (4, 32, kaxis, ASYM), (8, 32, PT, ASYM), key_outlier_frac=0.02,
           key_outlier_scale=12.0, seed=9)
    run_case(wl, [5000, 333], generic=False, global_combine=True, max_splits=max_splits)


@pytest.mark.parametrize("generic", [False, True], ids=["specialized", "generic"])
@pytest.mark.parametrize("case", FAST_CASES, ids=[c[0] for c in FAST_CASES])
def test_specialized_and_generic_kernels(case, generic):
    name, B, Hq, H, D, kc, vc, lens = case
    wl = W(name, B, Hq, H, D, kc, vc, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=7)
    run_case(wl, lens, generic=generic)


def _ord16(h):
    """fp16 values as integers whose differences count ulps (sign-magnitude -> ordered)."""
    u = np.asarray(h, np.float16).view(np.uint16).astype(np.int32)
    return np.where(u & 0x8000, -(u & 0x7FFF), u)


MAT_CASES = [CASES[0], CASES[6], CASES[7], CASES[11], CASES[14], CASES[15], FAST_CASES[2]]


@pytest.mark.parametrize("case", MAT_CASES, ids=[c[0] for c in MAT_CASES])
def test_materialized_baseline(case):
    """kvq_dequantize writes the oracle's dequantized cache rounded to fp16
    (within one fp16 ulp: the GPU rounds its one-rounding fp32 value, the oracle
    an exact one), and kvq_decode_attn_materialized over those rows agrees with
    the oracle's attention over the unrounded cache within the path's
    tolerance."""
    name, B, Hq, H, D, kc, vc, lens = case
    wl = W(name, B, Hq, H, D, kc, vc, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=21)
    T = max(max(lens), 1)
    cache = make_cache(wl, max_tokens=T)
    k, v = wl.layer_kv(0, "cpu", T=T)
    cache.kvq_prefill_quantize(0, k.cuda(), v.cuda(), lens)
    k16, v16 = cache.kvq_dequantize(0)
    q = wl.layer_query(0)
    scale = np.float32(1.0 / np.sqrt(D))
    out = cache.kvq_decode_attn_materialized(0, k16, v16, q.cuda(), scale=float(scale))
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    ok = oracle_tensor(k, lens, cache.tcap, wl.k, False)
    ov = oracle_tensor(v, lens, cache.tcap, wl.v, False)
    kh = oracle.dequant_tensor(ok, lens, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]))
    vh = oracle.dequant_tensor(ov, lens, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]))
    for gpu, ref, which in ((k16, kh, "k"), (v16, vh, "v")):
        g = gpu.cpu().numpy()
        for b, n in enumerate(lens):
            d = np.abs(_ord16(g[b, :, :n]) - _ord16(ref[b, :, :n].astype(np.float16)))
            assert d.size == 0 or d.max() <= 1, (which, b, d.max())
    ref_out = oracle.attention(kh, vh, q.float().numpy(), np.array(lens, np.int32), scale)
    err = rel_err_rows(out.cpu().numpy(), ref_out)
    for b, n in enumerate(lens):
        if n == 0:
            assert not out[b].any()
            err[b] = 0.0
    assert err.max() <= TOL, err.max()


GLOBAL_COMBINE_CASES = [CASES[0], CASES[11], FAST_CASES[0], FAST_CASES[2], FAST_CASES[6]]


@pytest.mark.parametrize("case", GLOBAL_COMBINE_CASES, ids=[c[0] for c in GLOBAL_COMBINE_CASES])
def test_global_workspace_combine(case):
    """The split-K partials merged through the global workspace and tickets
    (the path for more than 8 splits) agree with the oracle at every size."""
    name, B, Hq, H, D, kc, vc, lens = case
    wl = W(name, B, Hq, H, D, kc, vc, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=8)
    run_case(wl, lens, global_combine=True)


@pytest.mark.parametrize("case", CASES[:6] + CASES[12:], ids=[c[0] for c in CASES[:6] + CASES[12:]])
def test_parity_fp32_metadata(case):
    name, B, Hq, H, D, kc, vc, lens = case
    wl = W(name, B, Hq, H, D, kc, vc, seed=5)
    run_case(wl, lens, meta_f32=True)


def test_fp32_inputs_and_laplace_values():
    wl = W("f32", 2, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), torch.float32, value_dist="laplace", seed=9)
    run_case(wl, [640, 100])


def test_many_splits_and_ragged():
    wl = W("splits", 4, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), seed=11)
    run_case(wl, [3000, 1, 0, 1777], max_splits=64)


def test_two_level_combine_long_sequence():
    """One long sequence split into several hundred chunks: the partials merge
    in groups of 16 and then across groups."""
    wl = W("long", 1, 8, 1, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), seed=12)
    run_case(wl, [40000], max_splits=1024)


@pytest.mark.parametrize("kc,vc", [((4, 32, PC, ASYM), (4, 32, PT, ASYM)), ((2, 16, PC, SYM), (3, 16, PC, ASYM)),
                                   ((5, 64, PT, ASYM), (6, WHOLE, PT, ASYM))])
def test_append_equals_prefill(kc, vc):
    """Appending tokens one by one (with group sealing) gives bit-exactly the
    cache a prefill of the same tokens gives."""
    wl = W("app", 2, 4, 2, 64, kc, vc, torch.float32, seed=13)
    n0, steps = 20, 52
    T = n0 + steps
    k, v = wl.layer_kv(0, "cpu", T=T)
    cache = make_cache(wl, max_tokens=T)
    cache.kvq_prefill_quantize(0, k[:, :n0].contiguous().cuda(), v[:, :n0].contiguous().cuda(), [n0, n0])
    for s in range(steps):
        cache.kvq_append(0, k[:, n0 + s].contiguous().cuda(), v[:, n0 + s].contiguous().cuda())
    assert cache.kvq_get_lens(0) == [T, T]
    exp = cache.kvq_export(0)
    ref = make_cache(wl, max_tokens=T)
    ref.kvq_prefill_quantize(0, k.cuda(), v.cuda(), [T, T])
    exp2 = ref.kvq_export(0)
    torch.cuda.synchronize()
    for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens"):
        assert torch.equal(exp[key], exp2[key]), key
    for key in ("tail_k", "tail_v"):
        if exp[key] is not None:
            assert torch.equal(exp[key], exp2[key]), key
    ok = oracle_tensor(k, [T, T], cache.tcap, wl.k, False)
    assert_export_equal(exp, ok, wl.k, "k")
    q = wl.layer_query(0)
    scale = np.float32(0.125)
    out = cache.kvq_decode_attn(0, q.cuda(), scale=float(scale))
    ov = oracle_tensor(v, [T, T], cache.tcap, wl.v, False)
    ref_out = decode_ref(wl, ok, ov, [T, T], q, scale)
    assert rel_err_rows(out.cpu().numpy(), ref_out).max() <= TOL


def test_capacity_error_is_all_or_nothing():
    wl = W("cap", 2, 2, 2, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), seed=1)
    cache = make_cache(wl, max_tokens=40)
    k, v = wl.layer_kv(0, "cpu", T=40)
    cache.kvq_prefill_quantize(0, k.cuda(), v.cuda(), [40, 10])
    before = cache.kvq_export(0)
    with pytest.raises(kvq.KVQError) as e:
        cache.kvq_append(0, k[:, 0].contiguous().cuda(), v[:, 0].contiguous().cuda())
    assert e.value.status == 3
    after = cache.kvq_export(0)
    torch.cuda.synchronize()
    assert cache.kvq_get_lens(0) == [40, 10]
    for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens"):
        assert torch.equal(before[key], after[key])


# Full-precision recent window ("O Seu Cache KV Nao Tem um Problema de Bits...",
# section "O Imposto dos Sistemas e Por Que Nao E um Detalhe").
WINDOW_CASES = [
    ("w_mha64_k4pc_v4pt", 2, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), [300, 77], 64),
    ("w_mha128_kt_vt", 2, 2, 2, 128, (2, 32, PT, ASYM), (2, 32, PT, ASYM), [161, 40], 32),
    ("w_gqa8_256_pt", 1, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [700], 128),
    ("w_whole", 2, 4, 4, 64, (3, WHOLE, PT, ASYM), (3, WHOLE, PT, ASYM), [65, 140], 16),
    ("w_mha128_kc_vc", 1, 3, 3, 128, (2, 32, PC, ASYM), (2, 32, PC, ASYM), [1000], 128),
    ("w_gqa2_sym", 2, 4, 2, 128, (4, 64, PC, SYM), (4, 64, PT, SYM), [500, 3], 48),
    # Llama-2-13B's format with its 128-token window over long, ragged sequences:
    # the split weighs the window's fp16 tiles, so they spread over several warps
    ("w_llama_fmt_long", 3, 2, 2, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), [4113, 1500, 130], 128),
    ("w_wide_gqa_long", 1, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [9000], 1024),
]


@pytest.mark.parametrize("generic", [None, True], ids=["default", "generic"])
@pytest.mark.parametrize("case", WINDOW_CASES, ids=[c[0] for c in WINDOW_CASES])
def test_window_parity(case, generic):
    name, B, Hq, H, D, kc, vc, lens, window = case
    wl = W(name, B, Hq, H, D, kc, vc, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=17)
    run_case(wl, lens, generic=generic, window=window)


@pytest.mark.parametrize("max_splits", [0, 3], ids=["planned", "three_splits"])
@pytest.mark.parametrize("case", [c for c in WINDOW_CASES if c[0].endswith("_long")], ids=lambda c: c[0])
def test_window_parity_global_merge(case, max_splits):
    """The window's weighted split with the split-K partials merged through the
    global workspace, and with the splits capped (longer warp ranges, each
    holding more of the window)."""
    name, B, Hq, H, D, kc, vc, lens, window = case
    wl = W(name, B, Hq, H, D, kc, vc, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=18)
    run_case(wl, lens, global_combine=True, max_splits=max_splits, window=window)


@pytest.mark.parametrize("kc,vc,window", [((4, 32, PC, ASYM), (4, 32, PT, ASYM), 32),
                                          ((2, 16, PC, SYM), (3, 32, PT, ASYM), 64),
                                          ((5, 64, PT, ASYM), (6, WHOLE, PT, ASYM), 16)])
def test_window_append_equals_prefill(kc, vc, window):
    """Appending tokens one by one through a sliding window (fp16 rows, then
    group / block sealing from them) gives bit-exactly the cache a prefill of
    the same tokens gives, and the oracle's."""
    wl = W("wapp", 2, 4, 2, 64, kc, vc, torch.float32, seed=19)
    n0, steps = 20, 110
    T = n0 + steps
    k, v = wl.layer_kv(0, "cpu", T=T)
    cache = make_cache(wl, max_tokens=T, window=window)
    cache.kvq_prefill_quantize(0, k[:, :n0].contiguous().cuda(), v[:, :n0].contiguous().cuda(), [n0, n0])
    for s in range(steps):
        cache.kvq_append(0, k[:, n0 + s].contiguous().cuda(), v[:, n0 + s].contiguous().cuda())
    exp = cache.kvq_export(0)
    ref = make_cache(wl, max_tokens=T, window=window)
    ref.kvq_prefill_quantize(0, k.cuda(), v.cuda(), [T, T])
    exp2 = ref.kvq_export(0)
    torch.cuda.synchronize()
    for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens", "tail_k", "tail_v"):
        if exp[key] is not None:
            assert torch.equal(exp[key], exp2[key]), key
    ok = oracle_tensor(k, [T, T], cache.tcap, wl.k, False, window)
    ov = oracle_tensor(v, [T, T], cache.tcap, wl.v, False, window)
    assert_export_equal(exp, ok, wl.k, "k")
    assert_export_equal(exp, ov, wl.v, "v")
    q = wl.layer_query(0)
    scale = np.float32(0.125)
    out = cache.kvq_decode_attn(0, q.cuda(), scale=float(scale))
    ref_out = decode_ref(wl, ok, ov, [T, T], q, scale, window)
    assert rel_err_rows(out.cpu().numpy(), ref_out).max() <= TOL
