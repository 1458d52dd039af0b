"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (decode planned for the cache capacity), on sampled outputs the oracle
computes one (sequence, kv head) at a time.

Every registered workload variant (the GPT-2-small bits x group sweep under
both axis readings and its mixed K/V widths, the four Llama-2-13B axis
combinations, the wide-GQA K4/V8 and symmetric 6-bit settings with keys per
token or per channel, the serving mix) is built at full size for one layer on
the GPU (the layers of a workload are independent and identical in shape).
For a few (sequence, kv head) pairs the oracle quantizes that head's keys and
values (the same fp16 inputs), dequantizes them and computes the attention of
every query head that reads it.  Two error figures are checked against the
path's 1e-3: per (sequence, query head) row max|out - ref| / max|ref|, and
elementwise |out - ref| / max(|ref|, 1e-3 * max|ref of the row|).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_02_gb300 import build, kvq, synth

pytestmark = pytest.mark.gpu
TOL = 1e-3  # both figures

NAMES = [n for n in synth.WORKLOADS if n != "tiny"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


def _oracle_head(x_gpu, b, h, n, tc, tcap):
    """Oracle dequantized [T][D] of sequence b, kv head h (float64)."""
    bits, group, axis, mode = tc
    x = x_gpu[b:b + 1, :n, h:h + 1, :].float().cpu().numpy()
    lens = np.array([n], np.int32)
    # a whole-vector group spans every kv head of a token: quantize all heads, keep head h
    if group == kvq.WHOLE_VECTOR:
        x = x_gpu[b:b + 1, :n].float().cpu().numpy()
        q = oracle.quantize_tensor(x, lens, tcap, bits, group, axis, bool(mode))
        return oracle.dequant_tensor(q, lens, bits, group, axis, bool(mode))[0, h]
    q = oracle.quantize_tensor(x, lens, tcap, bits, group, axis, bool(mode))
    return oracle.dequant_tensor(q, lens, bits, group, axis, bool(mode))[0, 0]


def errors(got, ref):
    """(row-normalised max error, elementwise error with a 1e-3 row floor)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    rmax = np.abs(ref).max(axis=-1, keepdims=True)
    row = (d.max(axis=-1, keepdims=True) / rmax).max()
    elem = (d / np.maximum(np.abs(ref), 1e-3 * rmax)).max()
    return float(row), float(elem)


def _samples(B, H):
    return sorted({(0, 0), (B // 2, H - 1), (B - 1, H // 2)})


def _check(name, out, k, v, q, wl, lens, tcap, scale):
    rep = wl.q_heads // wl.kv_heads
    worst = (0.0, 0.0)
    for b, h in _samples(wl.batch, wl.kv_heads):
        n = int(lens[b])
        kh = _oracle_head(k, b, h, n, wl.k, tcap)
        vh = _oracle_head(v, b, h, n, wl.v, tcap)
        qs = q[b:b + 1, h * rep:(h + 1) * rep].float().cpu().numpy()
        ref = oracle.attention(kh[None, None], vh[None, None], qs, np.array([n], np.int32), scale)[0]
        row, elem = errors(out[b, h * rep:(h + 1) * rep], ref)
        worst = (max(worst[0], row), max(worst[1], elem))
        assert row <= TOL, (name, b, h, row)
    print(f"\n{name}: row {worst[0]:.2e} elementwise {worst[1]:.2e}")


def _build(name, window=0, kernel_bits=0):
    wl = synth.workload(name, layers=1)
    cap = wl.max_tokens + 8
    cfg = kvq.make_config(1, wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, cap, wl.k, wl.v,
                          recent_window=window)
    cache = kvq.KVQCache(cfg)
    if kernel_bits:
        cache.kvq_set_decode_kernel(kernel_bits)
    cache.kvq_set_decode_plan(cap)
    k, v = wl.layer_kv(0, "cuda", T=wl.max_tokens)
    cache.kvq_prefill_quantize(0, k, v, wl.lens)
    return wl, cache, k, v


# the workloads bench.py may time in one-warp CTAs (kvq_set_decode_kernel bit 2):
# the formats that have one-warp kernels
ONE_WARP = ["llama2_13b_kc_vt"]


@pytest.mark.parametrize("name", NAMES + [n + "@one_warp" for n in ONE_WARP])
def test_full_size_sampled_parity(name):
    base, _, shape = name.partition("@")
    wl, cache, k, v = _build(base, kernel_bits=4 if shape else 0)
    if shape:
        assert cache.kvq_decode_cta_warps() == 1
    q = wl.layer_query(0, 0, "cuda")
    scale = np.float32(1.0 / np.sqrt(wl.head_dim))
    out = cache.kvq_decode_attn(0, q, scale=float(scale))
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    _check(name, out.cpu().numpy(), k, v, q, wl, wl.lens, cache.tcap, scale)


@pytest.mark.parametrize("name", NAMES + [n + "@one_warp" for n in ONE_WARP])
def test_full_size_fused_step_sampled_parity(name):
    """One decode step of the benchmark's step graph at full size: the new
    token's append (fused into the decode launch when the format has a fused
    specialisation, else the append and decode kernels back to back), planned
    for the capacity, in four-warp CTAs and, for the formats that have them,
    one-warp CTAs.  Sampled (sequence, kv head) outputs against the oracle's
    quantization of the prefix plus the new token."""
    base, _, shape = name.partition("@")
    wl, cache, k, v = _build(base, kernel_bits=4 if shape else 0)
    if shape:
        assert cache.kvq_decode_cta_warps(True) == 1
    kn, vn = wl.step_kv(0, 0, "cuda")
    q = wl.layer_query(0, 1, "cuda")
    scale = np.float32(1.0 / np.sqrt(wl.head_dim))
    out = cache.kvq_append_decode_attn(0, kn, vn, q, scale=float(scale))
    assert cache.kvq_last_launches() in (1, 2)
    if cache.kvq_decode_kernel_specialized():
        assert cache.kvq_last_launches() == 1  # every specialised format has a fused form
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    cache.kvq_refresh_lens()  # the device lengths, advanced inside the launch
    lens = [int(x) + 1 for x in wl.lens]
    assert cache.kvq_get_lens(0) == lens
    T = wl.max_tokens
    kx = torch.empty((wl.batch, T + 1) + tuple(k.shape[2:]), dtype=k.dtype, device=k.device)
    vx = torch.empty_like(kx)
    for b in range(wl.batch):
        n = int(wl.lens[b])
        kx[b, :n], vx[b, :n] = k[b, :n], v[b, :n]
        kx[b, n], vx[b, n] = kn[b], vn[b]
    _check(name, out.cpu().numpy(), kx, vx, q, wl, lens, cache.tcap, scale)


@pytest.mark.parametrize("name", ["llama2_13b_kc_vt", "serving_mix", "wide_gqa_k4v8_kt", "llama2_13b_kc_vt@one_warp"])
def test_full_size_window_sampled_parity(name):
    """bench.py --window 128: the newest 128 tokens of both tensors stay fp16
    rows; the oracle quantizes the older tokens with the same window."""
    window = 128
    base, _, shape = name.partition("@")
    wl, cache, k, v = _build(base, window, kernel_bits=4 if shape else 0)
    q = wl.layer_query(0, 0, "cuda")
    scale = np.float32(1.0 / np.sqrt(wl.head_dim))
    out = cache.kvq_decode_attn(0, q, scale=float(scale))
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    rep = wl.q_heads // wl.kv_heads
    for b, h in _samples(wl.batch, wl.kv_heads):
        n = int(wl.lens[b])
        heads = []
        for x, tc in ((k, wl.k), (v, wl.v)):
            bits, group, axis, mode = tc
            xs = x[b:b + 1, :n, h:h + 1, :].float().cpu().numpy()
            oq = oracle.quantize_tensor(xs, np.array([n], np.int32), cache.tcap, bits, group, axis, bool(mode),
                                        False, window)
            heads.append(oracle.dequant_tensor(oq, [n], bits, group, axis, bool(mode), window)[0, 0])
        qs = q[b:b + 1, h * rep:(h + 1) * rep].float().cpu().numpy()
        ref = oracle.attention(heads[0][None, None], heads[1][None, None], qs, np.array([n], np.int32), scale)[0]
        row, elem = errors(out.cpu().numpy()[b, h * rep:(h + 1) * rep], ref)
        assert row <= TOL, (name, b, h, row)
