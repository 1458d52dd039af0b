"""kvq_decode_attn_static: decode attention for callers that cannot allocate.

Some callers cannot give the library device memory beyond what they planned
(a runtime whose device memory another component lays out once, a plugin that
must not call cudaMalloc).  kvq_decode_attn_static keeps the decode kernel's
scratch in an array compiled into libkvq; these tests call it through the C ABI
and check it against kvq_decode_attn, twice in a row (the array keeps the last
call's contents), and that a problem needing more scratch than the array holds
is refused.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from bit_quantized_kv_02_gb300 import build, kvq, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3


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
    k, v = wl.layer_kv(0, "cuda", T=T)
    cache.kvq_prefill_quantize(0, k, v, list(lens))
    return cache, wl


@pytest.mark.parametrize("shape", [
    (3, 4, 4, 64, [700, 65, 0], (4, 32, kvq.PER_CHANNEL, kvq.ASYM), (4, 32, kvq.PER_TOKEN, kvq.ASYM)),
    (2, 16, 2, 256, [900, 333], (4, 32, kvq.PER_TOKEN, kvq.ASYM), (8, 32, kvq.PER_TOKEN, kvq.ASYM)),
])
def test_static_scratch_matches_decode_twice(shape):
    B, Hq, H, D, lens, kc, vc = shape
    cache, wl = _cache(B, Hq, H, D, lens, kc, vc)
    for step in range(2):
        q = wl.layer_query(0, step, "cuda")
        ref = cache.kvq_decode_attn(0, q)
        got = cache.kvq_decode_attn_static(0, q)
        torch.cuda.synchronize()
        assert cache.kvq_device_status() == 0
        r = ref.double().cpu().numpy()
        g = got.double().cpu().numpy()
        err = np.abs(g - r).max(axis=-1) / np.maximum(np.abs(r).max(axis=-1), 1e-30)
        assert err.max() <= TOL, err.max()
        for b, n in enumerate(lens):
            if n == 0:
                assert not got[b].any()


def test_static_scratch_rejects_oversize():
    # 64 sequences x 32 query heads x 1024 splits x 132 floats is far beyond the 16 MiB array
    cfg = kvq.make_config(1, 64, 32, 8, 128, 4096, (2, 64, kvq.PER_CHANNEL, kvq.ASYM),
                          (2, 64, kvq.PER_TOKEN, kvq.ASYM), kvq.F16, 1024)
    cache = kvq.KVQCache(cfg)
    q = torch.zeros((64, 32, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        cache.kvq_decode_attn_static(0, q)
    assert e.value.status == 4
    assert "static array holds" in str(e.value)
