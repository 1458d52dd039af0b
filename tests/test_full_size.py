"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (decode planned for the cache capacity), on sampled outputs the oracle
computes one (sequence, kv head) at a time.

For each workload one layer is built at full size on the GPU; for a few
(sequence, kv head) pairs the oracle quantizes that head's keys and values
(the same fp16 inputs), dequantizes them and computes the attention of every
query head that reads it; the GPU output rows must agree within the path's
1e-3.  (The layers of the benchmark are independent and identical in shape.)
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_02_gb300 import build, kvq, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3

WORKLOADS = {
    "gpt2_small": lambda: synth.gpt2_small(layers=1),
    "gpt2_small_k6v4": lambda: synth.gpt2_small(kbits=6, vbits=4, kgroup=64, vgroup=64, kaxis=synth.PT,
                                                vaxis=synth.PT, layers=1),
    "llama2_13b": lambda: synth.llama2_13b(layers=1),
    "wide_gqa": lambda: synth.wide_gqa(),
    "serving_mix": lambda: synth.serving_mix(),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


def _oracle_head(x_gpu, b, h, n, tc, tcap):
    """Oracle dequantized [T][D] of sequence b, kv head h (float64)."""
    bits, group, axis, mode = tc
    x = x_gpu[b:b + 1, :n, h:h + 1, :].float().cpu().numpy()
    lens = np.array([n], np.int32)
    q = oracle.quantize_tensor(x, lens, tcap, bits, group, axis, bool(mode))
    return oracle.dequant_tensor(q, lens, bits, group, axis, bool(mode))[0, 0]


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_sampled_parity(name):
    wl = WORKLOADS[name]()
    B, Hq, H, D = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim
    rep = Hq // H
    cap = wl.max_tokens + 8
    cfg = kvq.make_config(1, B, Hq, H, D, cap, wl.k, wl.v)
    cache = kvq.KVQCache(cfg)
    cache.kvq_set_decode_plan(cap)
    k, v = wl.layer_kv(0, "cuda", T=wl.max_tokens)
    cache.kvq_prefill_quantize(0, k, v, wl.lens)
    q = wl.layer_query(0, 0, "cuda")
    scale = np.float32(1.0 / np.sqrt(D))
    out = cache.kvq_decode_attn(0, q, scale=float(scale))
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    out = out.cpu().numpy()
    tcap = cache.tcap
    samples = sorted({(0, 0), (B // 2, H - 1), (B - 1, H // 2)})
    for b, h in samples:
        n = int(wl.lens[b])
        kh = _oracle_head(k, b, h, n, wl.k, tcap)
        vh = _oracle_head(v, b, h, n, wl.v, tcap)
        qs = q[b:b + 1, h * rep:(h + 1) * rep].float().cpu().numpy()
        ref = oracle.attention(kh[None, None], vh[None, None], qs, np.array([n], np.int32), scale)[0]
        got = out[b, h * rep:(h + 1) * rep]
        err = np.abs(got - ref).max(axis=-1) / np.abs(ref).max(axis=-1)
        assert err.max() <= TOL, (name, b, h, err.max())


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_fused_step_sampled_parity(name):
    """One decode step of the benchmark's step graph at full size: the new
    token's append fused into the decode launch (one launch), planned for the
    capacity.  Sampled (sequence, kv head) outputs against the oracle's
    quantization of the prefix plus the new token."""
    wl = WORKLOADS[name]()
    B, Hq, H, D = wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim
    rep = Hq // H
    cap = wl.max_tokens + 8
    cfg = kvq.make_config(1, B, Hq, H, D, cap, wl.k, wl.v)
    cache = kvq.KVQCache(cfg)
    cache.kvq_set_decode_plan(cap)
    k, v = wl.layer_kv(0, "cuda", T=wl.max_tokens)
    cache.kvq_prefill_quantize(0, k, v, wl.lens)
    kn, vn = wl.step_kv(0, 0, "cuda")
    q = wl.layer_query(0, 1, "cuda")
    scale = np.float32(1.0 / np.sqrt(D))
    out = cache.kvq_append_decode_attn(0, kn, vn, q, scale=float(scale))
    assert cache.kvq_last_launches() == 1
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    cache.kvq_refresh_lens()  # the device lengths, advanced inside the launch
    assert cache.kvq_get_lens(0) == [int(x) + 1 for x in wl.lens]
    out = out.cpu().numpy()
    tcap = cache.tcap
    samples = sorted({(0, 0), (B // 2, H - 1), (B - 1, H // 2)})
    for b, h in samples:
        n = int(wl.lens[b])
        kx = torch.cat([k[b:b + 1, :n, h:h + 1, :], kn[b:b + 1, None, h:h + 1, :]], dim=1)
        vx = torch.cat([v[b:b + 1, :n, h:h + 1, :], vn[b:b + 1, None, h:h + 1, :]], dim=1)
        kh = _oracle_head(kx, 0, 0, n + 1, wl.k, tcap)
        vh = _oracle_head(vx, 0, 0, n + 1, wl.v, tcap)
        qs = q[b:b + 1, h * rep:(h + 1) * rep].float().cpu().numpy()
        ref = oracle.attention(kh[None, None], vh[None, None], qs, np.array([n + 1], np.int32), scale)[0]
        got = out[b, h * rep:(h + 1) * rep]
        err = np.abs(got - ref).max(axis=-1) / np.abs(ref).max(axis=-1)
        assert err.max() <= TOL, (name, b, h, err.max())
