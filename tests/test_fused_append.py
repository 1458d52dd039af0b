"""GPU parity of kvq_append_decode_attn (append fused into the decode launch).

Each decode step appends one token per sequence and then attends over the
whole cache.  The fused call must leave the cache exactly as kvq_append does
(codes, stored zero points / steps, fp16 tails and lengths bit-exact, which
the oracle's quantization of the same token sequence also pins), and its
output must match the separate kvq_append + kvq_decode_attn calls (same
arithmetic; only the per-warp operand scaling may differ by a power of two)
and the oracle's attention over the dequantized cache within 1e-3.
"""
import numpy as np
import pytest
import torch

from bit_quantized_kv_02_gb300 import build, kvq, synth
from test_gpu_parity import TOL, W, assert_export_equal, decode_ref, make_cache, oracle_tensor, rel_err_rows

pytestmark = pytest.mark.gpu
PT, PC, ASYM, SYM = kvq.PER_TOKEN, kvq.PER_CHANNEL, kvq.ASYM, kvq.SYM
SAME = 1e-5  # fused vs separate calls


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


CASES = [
    # name, B, Hq, H, D, k cfg, v cfg, prefill lengths, steps, launches (1: a fused specialisation
    # exists for the format, 2: the call runs the append and the decode kernels)
    ("mha64_k4pc_v4pt", 2, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), [300, 77], 40, 1),
    ("mha64_sym", 2, 2, 2, 64, (4, 32, PC, SYM), (2, 32, PT, SYM), [31, 150], 36, 2),
    ("mha64_k6pt_g64", 2, 2, 2, 64, (6, 64, PT, ASYM), (4, 64, PT, ASYM), [96, 33], 34, 1),
    ("mha64_k5_v7_g16", 1, 2, 2, 64, (5, 16, PC, ASYM), (7, 32, PT, ASYM), [129], 20, 2),
    ("mha128_kc_vt", 2, 3, 3, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), [95, 200], 40, 1),
    ("mha128_kc_vc", 2, 3, 3, 128, (2, 32, PC, ASYM), (2, 32, PC, ASYM), [95, 200], 40, 1),
    ("mha128_kt_vt", 2, 3, 3, 128, (2, 32, PT, ASYM), (2, 32, PT, ASYM), [95, 200], 40, 1),
    ("mha128_kt_vc", 2, 3, 3, 128, (2, 32, PT, ASYM), (2, 32, PC, ASYM), [63, 190], 40, 1),
    ("gqa8_256_sym6_pc", 1, 8, 1, 256, (6, 32, PC, SYM), (6, 32, PT, SYM), [333], 36, 1),
    ("mha128_kt_vc_g64", 2, 2, 2, 128, (2, 32, PT, ASYM), (3, 64, PC, ASYM), [60, 130], 70, 2),
    ("gqa4_128_empty", 3, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), [1000, 64, 0], 66, 1),
    ("gqa8_256_pt", 1, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [700], 20, 1),
    ("gqa8_256_pc", 1, 16, 2, 256, (4, 32, PC, ASYM), (8, 32, PT, ASYM), [650], 40, 1),
    ("gqa8_256_sym6", 1, 8, 1, 256, (6, 32, PT, SYM), (6, 32, PT, SYM), [333], 20, 1),
]


def step_tokens(wl, n0, steps):
    """Keys / values of the prefill and of each appended token: [B][n0+steps][H][D]."""
    T = max(n0) + steps
    return wl.layer_kv(0, "cpu", T=T)


def run_steps(wl, n0, steps, fused_kernel_bits=0, plan_tokens=0, check_every=10, window=0):
    T = max(n0) + steps
    k, v = step_tokens(wl, n0, steps)
    a = make_cache(wl, max_tokens=T, window=window)
    b = make_cache(wl, max_tokens=T, window=window)
    for c in (a, b):
        if fused_kernel_bits:
            c.kvq_set_decode_kernel(fused_kernel_bits)
        if plan_tokens:
            c.kvq_set_decode_plan(plan_tokens)
    # prefill each sequence's first n0[b] tokens (k is [B][T][H][D]; rows past
    # a sequence's length are ignored)
    kp, vp = k[:, :max(max(n0), 1)].contiguous().cuda(), v[:, :max(max(n0), 1)].contiguous().cuda()
    a.kvq_prefill_quantize(0, kp, vp, list(n0))
    b.kvq_prefill_quantize(0, kp, vp, list(n0))
    scale = np.float32(1.0 / np.sqrt(wl.head_dim))
    lens = list(n0)
    fused_launches = set()
    for s in range(steps):
        # token s of every sequence sits right after its own prefix
        kn = torch.stack([k[i, n0[i] + s] for i in range(wl.batch)]).contiguous().cuda()
        vn = torch.stack([v[i, n0[i] + s] for i in range(wl.batch)]).contiguous().cuda()
        q = wl.layer_query(0, step=s)
        a.kvq_append(0, kn, vn)
        out_a = a.kvq_decode_attn(0, q.cuda(), scale=float(scale))
        out_b = b.kvq_append_decode_attn(0, kn, vn, q.cuda(), scale=float(scale))
        fused_launches.add(b.kvq_last_launches())
        lens = [x + 1 for x in lens]
        torch.cuda.synchronize()
        assert a.kvq_device_status() == 0 and b.kvq_device_status() == 0
        assert rel_err_rows(out_b.cpu().numpy(), out_a.cpu().numpy()).max() <= SAME, s
        if s % check_every == check_every - 1 or s == steps - 1:
            # the cache a prefill of every token so far would hold (oracle)
            kk = torch.zeros((wl.batch, max(lens)) + tuple(k.shape[2:]), dtype=k.dtype)
            vv = torch.zeros_like(kk)
            for i in range(wl.batch):
                kk[i, :lens[i]] = k[i, :lens[i]]
                vv[i, :lens[i]] = v[i, :lens[i]]
            exp_b = b.kvq_export(0)
            exp_a = a.kvq_export(0)
            torch.cuda.synchronize()
            for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens", "tail_k", "tail_v"):
                if exp_a[key] is not None:
                    assert torch.equal(exp_a[key], exp_b[key]), (key, s)
            assert exp_b["lens"].cpu().tolist() == lens
            pad = b.tcap - kk.shape[1]
            kk = torch.nn.functional.pad(kk, (0, 0, 0, 0, 0, pad))
            vv = torch.nn.functional.pad(vv, (0, 0, 0, 0, 0, pad))
            ok = oracle_tensor(kk, lens, b.tcap, wl.k, False, window)
            ov = oracle_tensor(vv, lens, b.tcap, wl.v, False, window)
            assert_export_equal(exp_b, ok, wl.k, "k")
            assert_export_equal(exp_b, ov, wl.v, "v")
            ref = decode_ref(wl, ok, ov, lens, q, scale, window)
            assert rel_err_rows(out_b.cpu().numpy(), ref).max() <= TOL, s
    return fused_launches


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_append_matches_separate_calls(case):
    name, B, Hq, H, D, kc, vc, n0, steps, launches = case
    wl = W(name, B, Hq, H, D, kc, vc, torch.float32, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=5)
    assert run_steps(wl, n0, steps) == {launches}


# Full-precision recent window ("O Seu Cache KV Nao Tem um Problema de Bits...",
# section "O Imposto dos Sistemas e Por Que Nao E um Detalhe"): the fused step
# stores the new fp16 rows, and the block (per-token tensor, 16 tokens) or
# group (per-channel tensor) that leaves the window at that step is sealed
# inside the launch by the warp whose range holds it.  The steps cross
# several seals of each tensor.
WINDOW_CASES = [
    # name, B, Hq, H, D, k cfg, v cfg, prefill lengths, steps, window
    ("w_mha64_k4pc_v4pt", 2, 2, 2, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), [300, 77], 70, 32),
    ("w_mha64_k6pt_g64", 2, 2, 2, 64, (6, 64, PT, ASYM), (4, 64, PT, ASYM), [96, 33], 40, 16),
    ("w_mha128_kc_vt", 2, 3, 3, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), [95, 200], 70, 64),
    ("w_mha128_kt_vc", 2, 3, 3, 128, (2, 32, PT, ASYM), (2, 32, PC, ASYM), [63, 190], 70, 48),
    ("w_gqa4_128", 3, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), [1000, 64, 0], 70, 128),
    ("w_gqa8_256_pt", 1, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [700], 40, 32),
    ("w_gqa8_256_sym6_pc", 1, 8, 1, 256, (6, 32, PC, SYM), (6, 32, PT, SYM), [333], 70, 48),
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=[c[0] for c in WINDOW_CASES])
def test_fused_append_with_window(case):
    """One launch per step for every format with a fused specialisation; the
    cache bit-exact against the append kernel's (and the oracle's with the same
    window), the outputs as the separate calls' and within 1e-3 of the oracle."""
    name, B, Hq, H, D, kc, vc, n0, steps, window = case
    wl = W(name, B, Hq, H, D, kc, vc, torch.float32, key_outlier_frac=0.02, key_outlier_scale=12.0, seed=6)
    assert run_steps(wl, n0, steps, window=window, check_every=8) == {1}


@pytest.mark.parametrize("bits,launches", [(1, 2), (2, 1), (3, 2)], ids=["generic", "global_combine", "generic_global"])
def test_fused_append_other_kernels(bits, launches):
    """The generic (runtime-format) kernel has no fused form: the call runs
    the append and the decode kernels, with the same results."""
    wl = W("kinds", 2, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), torch.float32, seed=6)
    assert run_steps(wl, [200, 45], 40, fused_kernel_bits=bits) == {launches}


def test_fused_append_generic_format_falls_back():
    """A format without a compile-time specialisation (3-bit keys, 5-bit
    values) runs two kernels through the same call."""
    wl = W("f32meta", 2, 4, 4, 64, (3, 32, PC, ASYM), (5, 32, PT, ASYM), torch.float32, seed=10)
    assert run_steps(wl, [70, 20], 30) == {2}


def test_fused_append_planned_ahead_multi_wave():
    """A launch planned for more tokens than the cache holds (graph capture
    style) has CTAs past every sequence's end; many (sequence, head) pairs
    give several waves.  Every CTA still counts itself in exactly once."""
    wl = W("waves", 16, 8, 8, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), torch.float16, seed=7)
    n0 = [int(x) for x in np.random.default_rng(7).integers(900, 1500, 16)]
    assert run_steps(wl, n0, 33, plan_tokens=4000, check_every=16) == {1}


@pytest.mark.parametrize("fmt", ["mha_g32", "gqa4_g64"])
@pytest.mark.parametrize("bits", [0, 2], ids=["cluster_or_global", "global_combine"])
def test_fused_append_ragged_dead_chunks_many_steps(bits, fmt):
    """Ragged lengths (empty, one token, thousands) under a launch planned far
    beyond them: most CTAs of each (sequence, head) lie past its end and count
    themselves in as soon as they start, racing the CTAs that still hold work.
    Every CTA reads the old length before any CTA of its (sequence, head) can
    advance it, so over many steps the lengths, the cache and the outputs stay
    exactly those of the separate calls and the oracle."""
    if fmt == "mha_g32":  # formats with a fused specialisation (one launch per step)
        wl = W("ragged_dead", 6, 4, 4, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), torch.float16, seed=12)
    else:
        wl = W("ragged_dead", 6, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), torch.float16, seed=12)
    n0 = [2500, 40, 0, 700, 1, 129]
    assert run_steps(wl, n0, 64, fused_kernel_bits=bits, plan_tokens=6000, check_every=16) == {1}


def test_fused_append_falls_back_with_window():
    """A format with no fused specialisation (two queries per kv head at
    head_dim 64) and a full-precision window: the call runs the two kernels and
    gives the same results."""
    wl = W("win", 2, 4, 2, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), torch.float32, seed=8)
    T = 200
    k, v = wl.layer_kv(0, "cpu", T=T)
    a = make_cache(wl, max_tokens=T, window=32)
    b = make_cache(wl, max_tokens=T, window=32)
    for c in (a, b):
        c.kvq_prefill_quantize(0, k[:, :100].contiguous().cuda(), v[:, :100].contiguous().cuda(), [100, 100])
    for s in range(40):
        kn, vn = k[:, 100 + s].contiguous().cuda(), v[:, 100 + s].contiguous().cuda()
        q = wl.layer_query(0, step=s).cuda()
        a.kvq_append(0, kn, vn)
        out_a = a.kvq_decode_attn(0, q)
        out_b = b.kvq_append_decode_attn(0, kn, vn, q)
        assert b.kvq_last_launches() == 2
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b)
    ea, eb = a.kvq_export(0), b.kvq_export(0)
    for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens", "tail_k", "tail_v"):
        if ea[key] is not None:
            assert torch.equal(ea[key], eb[key]), key


def test_fused_append_graph_replay():
    """One captured fused step replayed: the device lengths advance at every
    replay exactly as with eager calls (kvq_refresh_lens brings them back)."""
    wl = W("graph", 4, 4, 4, 64, (4, 32, PC, ASYM), (4, 32, PT, ASYM), torch.float16, seed=9)
    T = 400
    k, v = wl.layer_kv(0, "cpu", T=T)
    n0 = [250, 31, 100, 7]
    a = make_cache(wl, max_tokens=T)
    b = make_cache(wl, max_tokens=T)
    kn, vn = k[:, 300].contiguous().cuda(), v[:, 300].contiguous().cuda()
    q = wl.layer_query(0).cuda()
    st = torch.cuda.Stream()
    for c in (a, b):
        c.kvq_prefill_quantize(0, k[:, :250].contiguous().cuda(), v[:, :250].contiguous().cuda(), n0)
        c.kvq_set_decode_plan(T)
    out_b = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        b.kvq_append_decode_attn(0, kn, vn, q, out=out_b, stream=st)
    torch.cuda.synchronize()
    assert b.kvq_last_launches() == 1
    b.kvq_refresh_lens()  # the capture itself launched nothing
    for s in range(45):
        out_a = a.kvq_append_decode_attn(0, kn, vn, q)
        g.replay()
        torch.cuda.synchronize()
        assert rel_err_rows(out_b.cpu().numpy(), out_a.cpu().numpy()).max() <= SAME, s
    b.kvq_refresh_lens()
    ea, eb = a.kvq_export(0), b.kvq_export(0)
    torch.cuda.synchronize()
    for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens", "tail_k", "tail_v"):
        if ea[key] is not None:
            assert torch.equal(ea[key], eb[key]), key
    assert eb["lens"].cpu().tolist() == [x + 45 for x in n0]


def test_fused_append_near_half_integer_quotients():
    """Appended per-token values whose quotients (x - zero) / step sit on and
    around half-integers (offsets from 0 up to 1e-3, across the 2^-12 cutoff
    below which the IEEE division decides the rounding): codes equal the
    oracle's and the append kernel's bit for bit."""
    import oracle

    B, Hq, H, D, G = 2, 4, 4, 64, 32
    wl = W("near_half", B, Hq, H, D, (4, 32, PC, ASYM), (4, G, PT, ASYM), torch.float32, seed=11)
    n0, steps = 40, 40
    T = n0 + steps
    k, v = wl.layer_kv(0, "cpu", T=T)
    v = v.clone()
    rng = np.random.default_rng(11)
    deltas = [0.0, 2**-22, -2**-22, 2**-14, -2**-14, 2**-13, -2**-13, 2**-12, -2**-12, 2**-11, -2**-11,
              2**-9, -2**-9, 1e-3, -1e-3]
    for t in range(n0, T):
        for b in range(B):
            for h in range(H):
                row = np.zeros(D, np.float32)
                for j in range(D // G):
                    row[j * G + 1] = np.float32(rng.uniform(0.5, 8.0))  # each group spans [0, M]
                meta = oracle.quantize_tensor(row.reshape(1, 1, 1, D), np.array([1], np.int32), 16, 4, G, PT)["meta"]
                for j in range(D // G):
                    z, s = float(meta[j][0]), float(meta[j][1])
                    assert z == 0.0
                    for i in range(2, G):
                        kk = int(rng.integers(0, 13))
                        row[j * G + i] = np.float32((kk + 0.5 + deltas[(i + t) % len(deltas)]) * s)
                v[b, t, h] = torch.from_numpy(row)
    a = make_cache(wl, max_tokens=T)
    b_ = make_cache(wl, max_tokens=T)
    for c in (a, b_):
        c.kvq_prefill_quantize(0, k[:, :n0].contiguous().cuda(), v[:, :n0].contiguous().cuda(), [n0] * B)
    q = wl.layer_query(0).cuda()
    for t in range(n0, T):
        kn, vn = k[:, t].contiguous().cuda(), v[:, t].contiguous().cuda()
        a.kvq_append(0, kn, vn)
        b_.kvq_append_decode_attn(0, kn, vn, q)
        assert b_.kvq_last_launches() == 1
    ea, eb = a.kvq_export(0), b_.kvq_export(0)
    torch.cuda.synchronize()
    for key in ("codes_k", "codes_v", "meta_k", "meta_v", "lens", "tail_k"):
        assert torch.equal(ea[key], eb[key]), key
    ov = oracle_tensor(v, [T] * B, b_.tcap, wl.v, False)
    ok = oracle_tensor(k, [T] * B, b_.tcap, wl.k, False)
    assert_export_equal(eb, ov, wl.v, "v")
    assert_export_equal(eb, ok, wl.k, "k")
