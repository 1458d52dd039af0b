"""Host-side tests of the C ABI (no GPU): the library loads, exports every
symbol include/kvq.h declares, validates arguments before touching CUDA, and
its byte accounting agrees with the oracle's size terms."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from bit_quantized_kv_02_gb300 import build, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(kvq.LIB_PATH):
        build.build()
    return kvq.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(kvq.EXPORTED)


def test_status_strings(L):
    assert kvq.kvq_status_string(0) == "ok"
    assert "capacity" in kvq.kvq_status_string(3)


def _cfg(**kw):
    base = dict(layers=2, batch=3, q_heads=8, kv_heads=2, head_dim=64, max_tokens=100,
                k=(4, 32, kvq.PER_CHANNEL, kvq.ASYM), v=(4, 32, kvq.PER_TOKEN, kvq.ASYM))
    base.update(kw)
    return kvq.make_config(base["layers"], base["batch"], base["q_heads"], base["kv_heads"], base["head_dim"],
                           base["max_tokens"], base["k"], base["v"], base.get("meta_dtype", 0), base.get("max_splits", 0),
                           base.get("recent_window", 0), base.get("rope_theta", 0.0))


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2), (dict(q_heads=6), 2), (dict(q_heads=7), 1), (dict(batch=2000), 2),
    (dict(k=(1, 32, 1, 0)), 1), (dict(k=(9, 32, 1, 0)), 1), (dict(k=(4, 48, 1, 0)), 2),
    (dict(v=(4, 48, 0, 0)), 2), (dict(v=(4, 128, 0, 0)), 2), (dict(k=(4, -1, 1, 0)), 1),
    (dict(k=(4, 32, 2, 0)), 1), (dict(k=(4, 32, 1, 5)), 1), (dict(meta_dtype=3), 1), (dict(layers=0), 1),
    (dict(kv_heads=16, head_dim=256, v=(4, -1, 0, 0), q_heads=16), 2),
    (dict(recent_window=8), 1), (dict(recent_window=-16), 1), (dict(recent_window=1040), 1),
    (dict(rope_theta=-1.0), 1), (dict(rope_theta=0.5), 1), (dict(rope_theta=float("inf")), 1),
    (dict(rope_theta=float("nan")), 1), (dict(rope_theta=10000.0, max_tokens=(1 << 24) + 1), 2),
])
def test_config_validation(L, kw, status):
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_cache_bytes(_cfg(**kw))
    assert e.value.status == status


def test_capacity_and_buffer_checks(L):
    cfg = _cfg()
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_cache_bytes(cfg, [10, 101, 5])
    assert e.value.status == 3
    b = kvq.kvq_cache_bytes(cfg)
    h = ctypes.c_void_p()
    # a too-small buffer is rejected before any CUDA call (the pointer is never touched)
    st = L.kvq_cache_create(ctypes.byref(cfg), ctypes.c_void_p(1 << 20), b.alloc - 1, None, ctypes.byref(h))
    assert st == 4
    st = L.kvq_cache_create(ctypes.byref(cfg), ctypes.c_void_p((1 << 20) + 8), b.alloc, None, ctypes.byref(h))
    assert st == 1
    assert L.kvq_cache_create(ctypes.byref(cfg), None, b.alloc, None, ctypes.byref(h)) == 1
    assert L.kvq_decode_attn(None, 0, None, 0, 0.0, None, None) == 1
    assert L.kvq_append(None, 0, None, None, 0, None) == 1
    assert L.kvq_append_decode_attn(None, 0, None, None, 0, None, 0, 0.0, None, None) == 1


def test_decode_kernel_choice_without_a_handle(L):
    """The decode-kernel switches and queries refuse a null handle before any CUDA call."""
    for which in (0, 4, 7, 8, -1):
        assert L.kvq_set_decode_kernel(None, which) == 1
    assert L.kvq_decode_cta_warps(None, 0) == 0
    assert L.kvq_decode_cta_warps(None, 1) == 0
    assert L.kvq_decode_kernel_specialized(None) == 0


@pytest.mark.parametrize("window", [0, 64])
@pytest.mark.parametrize("k,v,meta_f32", [
    ((4, 32, 1, 0), (4, 32, 0, 0), 0), ((2, 64, 1, 0), (2, 64, 0, 0), 0), ((6, 64, 0, 0), (4, 64, 0, 0), 0),
    ((3, -1, 0, 1), (8, 128, 1, 1), 1), ((5, 16, 1, 0), (7, -1, 0, 0), 0),
])
def test_byte_accounting_matches_oracle(L, k, v, meta_f32, window):
    H, D, B, layers = 3, 128, 4, 2
    cfg = _cfg(layers=layers, batch=B, kv_heads=H, q_heads=H * 2, head_dim=D, max_tokens=300, k=k, v=v,
               meta_dtype=meta_f32, recent_window=window)
    lens = [0, 17, 200, 300]
    b = kvq.kvq_cache_bytes(cfg, lens)
    pk, mk, tk = oracle.tensor_bytes(B, H, D, np.array(lens), k[0], k[1], k[2], bool(k[3]), bool(meta_f32), window)
    pv, mv, tv = oracle.tensor_bytes(B, H, D, np.array(lens), v[0], v[1], v[2], bool(v[3]), bool(meta_f32), window)
    assert b.packed == layers * (pk + pv)
    assert b.metadata == layers * (mk + mv)
    assert b.tail == layers * (tk + tv)
    assert b.elements == oracle.cache_elements(layers, sum(lens), H, D)
    assert b.total == b.packed + b.metadata + b.tail + b.workspace
    assert b.alloc >= b.packed + b.metadata
