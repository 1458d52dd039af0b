"""kvq_decode_attn_static: decode attention for callers that cannot allocate.

Some callers cannot give the library device memory beyond what they planned
(a runtime whose device memory another component lays out once, a plugin that
must not call cudaMalloc).  kvq_decode_attn_static keeps the decode kernel's
scratch (split-K partials, group partials and combine tickets) in an array
compiled into libkvq.  These tests call it through the C ABI, twice in a row
(the array keeps the last call's contents), and check its output against
kvq_decode_attn and against the oracle's attention over the same quantized
cache.  The shapes reach every part of the array: a cluster merge (no
partials in the array), the one-group ticket merge and the two-level merge
(more than 16 splits: chunk partials, group partials and both ticket kinds).
A problem needing more scratch than the array holds, and an infinite
softmax scale, are refused without a launch.  This file is collected last on
purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_02_gb300 import build, kvq, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3
PT, PC, ASYM = kvq.PER_TOKEN, kvq.PER_CHANNEL, kvq.ASYM


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


def _cache(B, Hq, H, D, lens, kc, vc, max_splits=0, seed=4):
    wl = synth.Workload("na", 1, B, Hq, H, D, list(lens), kc, vc, torch.float16, key_outlier_frac=0.02,
                        key_outlier_scale=10.0, seed=seed)
    T = max(lens)
    cfg = kvq.make_config(1, B, Hq, H, D, T, kc, vc, kvq.F16, max_splits)
    cache = kvq.KVQCache(cfg)
    k, v = wl.layer_kv(0, "cpu", T=T)
    cache.kvq_prefill_quantize(0, k.cuda(), v.cuda(), list(lens))
    return cache, wl, k, v


def _oracle_out(wl, k, v, lens, tcap, q, scale):
    ln = np.array(lens, np.int32)
    ok = oracle.quantize_tensor(k.float().numpy(), ln, tcap, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]))
    ov = oracle.quantize_tensor(v.float().numpy(), ln, tcap, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]))
    kh = oracle.dequant_tensor(ok, ln, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]))
    vh = oracle.dequant_tensor(ov, ln, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]))
    return oracle.attention(kh, vh, q.float().numpy(), ln, scale)


def _rel_rows(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref).max(axis=-1) / np.maximum(np.abs(ref).max(axis=-1), 1e-30)


SHAPES = [
    # B, Hq, H, D, lens, k cfg, v cfg, max_splits
    ("mha64_short", 3, 4, 4, 64, [700, 65, 0], (4, 32, PC, ASYM), (4, 32, PT, ASYM), 0),
    ("gqa8_256", 2, 16, 2, 256, [900, 333], (4, 32, PT, ASYM), (8, 32, PT, ASYM), 0),
    # one long sequence and one short: about 60 splits of the long one, merged
    # in groups of 16 and then across the groups
    ("two_level", 2, 8, 2, 128, [8000, 150], (2, 32, PC, ASYM), (2, 32, PT, ASYM), 64),
]


@pytest.mark.parametrize("global_combine", [False, True], ids=["default_merge", "global_merge"])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_static_scratch_matches_decode_and_oracle_twice(shape, global_combine):
    _, B, Hq, H, D, lens, kc, vc, max_splits = shape
    cache, wl, k, v = _cache(B, Hq, H, D, lens, kc, vc, max_splits)
    if global_combine:
        cache.kvq_set_decode_kernel(2)  # merge through the scratch array even where a cluster could
    scale = np.float32(1.0 / np.sqrt(D))
    for step in range(2):
        q = wl.layer_query(0, step)
        ref = cache.kvq_decode_attn(0, q.cuda(), scale=float(scale))
        got = cache.kvq_decode_attn_static(0, q.cuda(), scale=float(scale))
        torch.cuda.synchronize()
        assert cache.kvq_device_status() == 0
        g = got.double().cpu().numpy()
        assert _rel_rows(g, ref.double().cpu().numpy()).max() <= TOL
        want = _oracle_out(wl, k, v, lens, cache.tcap, q, scale)
        err = _rel_rows(g, want)
        for b, n in enumerate(lens):
            if n == 0:
                assert not got[b].any()
                err[b] = 0.0
        assert err.max() <= TOL, (step, err.max())


def test_static_scratch_rejects_oversize():
    # 64 sequences x 32 query heads x 1024 splits x 132 floats is far beyond the 16 MiB array
    cfg = kvq.make_config(1, 64, 32, 8, 128, 4096, (2, 64, PC, ASYM), (2, 64, PT, ASYM), kvq.F16, 1024)
    cache = kvq.KVQCache(cfg)
    q = torch.zeros((64, 32, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        cache.kvq_decode_attn_static(0, q)
    assert e.value.status == 4
    assert "static array holds" in str(e.value)


def test_static_scratch_rejects_non_finite_scale():
    cache, wl, _, _ = _cache(1, 4, 4, 64, [100], (4, 32, PC, ASYM), (4, 32, PT, ASYM))
    q = wl.layer_query(0).cuda()
    # (a scale <= 0, or NaN, selects the default 1/sqrt(head_dim); +inf is an error)
    with pytest.raises(kvq.KVQError) as e:
        cache.kvq_decode_attn_static(0, q, scale=float("inf"))
    assert e.value.status == 1
    with pytest.raises(kvq.KVQError) as e:
        cache.kvq_decode_attn(0, q, scale=float("inf"))
    assert e.value.status == 1
