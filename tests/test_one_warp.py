"""GPU parity of the one-warp-CTA decode kernels (kvq_set_decode_kernel bit 2).

With bit 2 set, a format that has a one-warp specialisation (2-bit MHA at
head_dim 128, keys per channel / values per token, groups of 32: the
Llama-2-13B-shaped workload's format) launches one warp per CTA: every CTA
streams one token range and the ranges of a (sequence, head) merge through the
global workspace.  The launch shape must not change the result: decode
attention within 1e-3 of the oracle's attention over the same dequantized
cache per (sequence, query head) row, the fused decode step bit-exact with the
separate append (cache and lengths) and within 1e-3 of the oracle, and the
outputs within 1e-4 of the four-warp kernels' (other range boundaries, so the
fp32 partial sums round at other places).
"""
import numpy as np
import pytest
import torch

from bit_quantized_kv_02_gb300 import build, kvq
from test_fused_append import run_steps
from test_gpu_parity import TOL, W, decode_ref, make_cache, oracle_tensor, rel_err_rows, run_case

pytestmark = pytest.mark.gpu
PT, PC, ASYM = kvq.PER_TOKEN, kvq.PER_CHANNEL, kvq.ASYM
ONE_WARP = 4
NEAR = 1e-4
FMT = ((2, 32, PC, ASYM), (2, 32, PT, ASYM))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


@pytest.mark.parametrize("lens,max_splits", [([1500, 77, 0, 641], 0), ([4113, 4113], 0), ([9000, 33], 64)],
                         ids=["ragged", "equal", "two_level"])
def test_one_warp_decode_parity(lens, max_splits):
    wl = W("one_warp", len(lens), 6, 6, 128, *FMT, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=21)
    T = max(lens)
    k, v = wl.layer_kv(0, "cpu", T=T)
    caches = []
    for bits in (ONE_WARP, 0):
        c = make_cache(wl, max_tokens=T, max_splits=max_splits)
        c.kvq_set_decode_kernel(bits)
        assert c.kvq_decode_kernel_specialized()
        c.kvq_prefill_quantize(0, k.cuda(), v.cuda(), lens)
        caches.append(c)
    q = wl.layer_query(0)
    scale = np.float32(1.0 / np.sqrt(128))
    outs = []
    for c in caches:
        o = c.kvq_decode_attn(0, q.cuda(), scale=float(scale))
        torch.cuda.synchronize()
        assert c.kvq_device_status() == 0
        outs.append(o.cpu().numpy())
    ok = oracle_tensor(k, lens, caches[0].tcap, wl.k, False)
    ov = oracle_tensor(v, lens, caches[0].tcap, wl.v, False)
    ref = decode_ref(wl, ok, ov, lens, q, scale)
    live = np.array(lens) > 0
    assert rel_err_rows(outs[0][live], ref[live]).max() <= TOL
    assert rel_err_rows(outs[0][live], outs[1][live]).max() <= NEAR
    assert not outs[0][~live].any()
    # the allocation-free entry point runs the same launch
    st = caches[0].kvq_decode_attn_static(0, q.cuda(), scale=float(scale))
    torch.cuda.synchronize()
    assert rel_err_rows(st.cpu().numpy()[live], outs[0][live]).max() <= NEAR


def test_one_warp_global_merge_bits_combined():
    """Bit 2 with bit 1 (global merge, which one-warp CTAs use anyway)."""
    wl = W("one_warp_g", 3, 4, 4, 128, *FMT, seed=22)
    c = run_case(wl, [700, 1234, 5], global_combine=True)
    del c


@pytest.mark.parametrize("n0,plan", [([300, 77, 1000], 0), ([2500, 40, 0, 700, 1, 129], 6000)],
                         ids=["ragged", "planned_ahead_dead_chunks"])
def test_one_warp_fused_steps(n0, plan):
    """Decode steps through kvq_append_decode_attn with one-warp CTAs: one
    launch per step, the cache bit-exact with kvq_append's and the oracle's,
    the outputs as the separate calls' and within 1e-3 of the oracle; with a
    launch planned far past the lengths, CTAs past a sequence's end count
    themselves in and leave, and the lengths still advance once per step."""
    wl = W("one_warp_fused", len(n0), 4, 4, 128, *FMT, torch.float32, key_outlier_frac=0.02,
           key_outlier_scale=12.0, seed=23)
    assert run_steps(wl, n0, 40, fused_kernel_bits=ONE_WARP, plan_tokens=plan, check_every=13) == {1}


def test_one_warp_window_decode_and_steps():
    """A 64-token full-precision window: decode over packed tiles and fp16 rows,
    then decode steps whose seals move blocks out of the window."""
    window = 64
    wl = W("one_warp_win", 3, 4, 4, 128, *FMT, torch.float32, key_outlier_frac=0.02, key_outlier_scale=12.0,
           seed=24)
    lens = [900, 130, 64]
    T = max(lens)
    k, v = wl.layer_kv(0, "cpu", T=T)
    c = make_cache(wl, max_tokens=T, window=window)
    c.kvq_set_decode_kernel(ONE_WARP)
    c.kvq_prefill_quantize(0, k.cuda(), v.cuda(), lens)
    q = wl.layer_query(0)
    scale = np.float32(1.0 / np.sqrt(128))
    out = c.kvq_decode_attn(0, q.cuda(), scale=float(scale))
    torch.cuda.synchronize()
    ok = oracle_tensor(k, lens, c.tcap, wl.k, False, window)
    ov = oracle_tensor(v, lens, c.tcap, wl.v, False, window)
    assert rel_err_rows(out.cpu().numpy(), decode_ref(wl, ok, ov, lens, q, scale, window)).max() <= TOL
    assert run_steps(wl, [200, 63, 500], 36, fused_kernel_bits=ONE_WARP, window=window, check_every=12) == {1}


def test_cta_warps_query():
    """kvq_decode_cta_warps reports the shape each call launches: one warp only
    where the format has that specialisation and bit 2 asks for it; 0 for the
    decode step when it runs two kernels (the generic kernel has no fused form)."""
    wl = W("shape", 2, 4, 4, 128, *FMT, seed=25)
    c = make_cache(wl, max_tokens=64)
    assert (c.kvq_decode_cta_warps(), c.kvq_decode_cta_warps(True)) == (4, 4)
    c.kvq_set_decode_kernel(ONE_WARP)
    assert (c.kvq_decode_cta_warps(), c.kvq_decode_cta_warps(True)) == (1, 1)
    c.kvq_set_decode_kernel(ONE_WARP | 1)  # the generic kernel: four warps, no fused step
    assert (c.kvq_decode_cta_warps(), c.kvq_decode_cta_warps(True)) == (4, 0)
    other = make_cache(W("other", 2, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), seed=25), max_tokens=64)
    other.kvq_set_decode_kernel(ONE_WARP)  # no one-warp specialisation for this format
    assert (other.kvq_decode_cta_warps(), other.kvq_decode_cta_warps(True)) == (4, 4)
