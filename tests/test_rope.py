"""GPU parity of pre-RoPE key quantization.

"O Seu Cache KV Nao Tem um Problema de Bits. Tem um Problema de Geometria",
sections "Embebedos Rotatorios Complicam as Chaves" and "O Que Fazer Com
Isso", item 2: keys are quantized before the rotary position embedding and
rotated after dequantization.  With kvq_config.rope_theta > 0 the cache holds
the pre-RoPE keys (codes, metadata and fp16 tails bit-exact against the
oracle's quantization of the same keys) and decode attention turns every
dequantized key by its token's angles; the reference is the oracle's
attention over its dequantized keys rotated by oracle.rope, within the
path's 1e-3 per (sequence, query head) row.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_kv_02_gb300 import build, kvq, synth
from test_gpu_parity import TOL, assert_export_equal, oracle_tensor, rel_err_rows

pytestmark = pytest.mark.gpu
PT, PC, ASYM, SYM = kvq.PER_TOKEN, kvq.PER_CHANNEL, kvq.ASYM, kvq.SYM


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    kvq.lib()


CASES = [
    # name, B, Hq, H, D, k cfg, v cfg, lengths, rope base
    ("mha128_kc_vt_tail", 2, 4, 4, 128, (2, 32, PC, ASYM), (2, 32, PT, ASYM), [1000, 77], 10000.0),
    ("mha64_kt_vc", 2, 2, 2, 64, (4, 32, PT, ASYM), (4, 32, PC, ASYM), [640, 300], 10000.0),
    ("gqa4_128_kc_g64", 2, 8, 2, 128, (2, 64, PC, ASYM), (2, 64, PT, ASYM), [2500, 0], 500000.0),
    ("gqa8_256_kt", 1, 16, 2, 256, (4, 32, PT, ASYM), (8, 32, PT, ASYM), [1500], 10000.0),
    ("gqa8_256_sym6_kc", 1, 8, 1, 256, (6, 32, PC, SYM), (6, 32, PT, SYM), [700], 1000000.0),
    ("mha64_k3_v5_g16_whole", 2, 4, 4, 64, (3, kvq.WHOLE_VECTOR, PT, ASYM), (5, 16, PC, ASYM), [333, 48],
     10000.0),
]


def _rope_ref(wl, ok, ov, lens, q_cpu, scale, base):
    kh = oracle.dequant_tensor(ok, lens, wl.k[0], wl.k[1], wl.k[2], bool(wl.k[3]))
    vh = oracle.dequant_tensor(ov, lens, wl.v[0], wl.v[1], wl.v[2], bool(wl.v[3]))
    kh = oracle.rope(kh, lens, base)
    return oracle.attention(kh, vh, q_cpu.float().numpy(), np.array(lens, np.int32), scale)


def _workload(name, B, Hq, H, D, kc, vc, seed):
    return synth.Workload(name, 1, B, Hq, H, D, [1], kc, vc, torch.float16, key_outliers_per_head=2,
                          key_outlier_scale=12.0, seed=seed)


@pytest.mark.parametrize("which", [0, 1, 2], ids=["default", "generic", "global_merge"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rope_decode_parity(case, which):
    """which: kvq_set_decode_kernel bits (0: the compile-time rotary
    specialisation where the format has one, else the runtime-format rotary
    kernel; 1: always the runtime-format kernel; 2: merge through the global
    workspace)."""
    name, B, Hq, H, D, kc, vc, lens, base = case
    wl = _workload(name, B, Hq, H, D, kc, vc, seed=21)
    T = max(max(lens), 1)
    cfg = kvq.make_config(1, B, Hq, H, D, T, kc, vc, rope_theta=base)
    cache = kvq.KVQCache(cfg)
    if which:
        cache.kvq_set_decode_kernel(which)
    if which & 1:
        assert not cache.kvq_decode_kernel_specialized()
    elif name == "mha128_kc_vt_tail":
        assert cache.kvq_decode_kernel_specialized()  # the Llama-2-13B format has a rotary specialisation
    k, v = wl.layer_kv(0, "cpu", T=T)
    cache.kvq_prefill_quantize(0, k.cuda(), v.cuda(), lens)
    exp = cache.kvq_export(0)
    torch.cuda.synchronize()
    ok = oracle_tensor(k, lens, cache.tcap, kc, False)
    ov = oracle_tensor(v, lens, cache.tcap, vc, False)
    assert_export_equal(exp, ok, kc, "k")  # the cache holds the pre-RoPE keys as given
    assert_export_equal(exp, ov, vc, "v")
    q = wl.layer_query(0)
    scale = np.float32(1.0 / np.sqrt(D))
    out = cache.kvq_decode_attn(0, q.cuda(), scale=float(scale))
    torch.cuda.synchronize()
    assert cache.kvq_device_status() == 0
    ref = _rope_ref(wl, ok, ov, lens, q, scale, base)
    err = rel_err_rows(out.cpu().numpy(), ref)
    for b, n in enumerate(lens):
        if n == 0:
            assert not out[b].any()
            err[b] = 0.0
    assert err.max() <= TOL, err.max()
    # the rotation matters: attention over unrotated keys is far from the output
    kh = oracle.dequant_tensor(ok, lens, kc[0], kc[1], kc[2], bool(kc[3]))
    vh = oracle.dequant_tensor(ov, lens, vc[0], vc[1], vc[2], bool(vc[3]))
    plain = oracle.attention(kh, vh, q.float().numpy(), np.array(lens, np.int32), scale)
    busy = [b for b, n in enumerate(lens) if n > 1]
    assert rel_err_rows(out.cpu().numpy()[busy], plain[busy]).max() > 1e-2


def test_rope_decode_steps_and_materialized():
    """Decode steps through kvq_append_decode_attn (the append and the rotary
    decode kernel back to back) over a growing cache: every step's output
    against the oracle over the pre-RoPE keys rotated at their positions, and
    the materialised baseline (dequantize to fp16 rows, then decode) rotating
    the same keys."""
    B, Hq, H, D = 2, 8, 2, 128
    kc, vc = (2, 32, PC, ASYM), (2, 32, PT, ASYM)
    wl = _workload("steps", B, Hq, H, D, kc, vc, seed=22)
    n0, steps, base = [200, 31], 40, 10000.0
    T = max(n0) + steps
    k, v = wl.layer_kv(0, "cpu", T=T)
    cache = kvq.KVQCache(kvq.make_config(1, B, Hq, H, D, T, kc, vc, rope_theta=base))
    cache.kvq_prefill_quantize(0, k[:, :max(n0)].contiguous().cuda(), v[:, :max(n0)].contiguous().cuda(), n0)
    scale = np.float32(1.0 / np.sqrt(D))
    lens = list(n0)
    for s in range(steps):
        kn = torch.stack([k[i, n0[i] + s] for i in range(B)]).contiguous()
        vn = torch.stack([v[i, n0[i] + s] for i in range(B)]).contiguous()
        q = wl.layer_query(0, step=s)
        out = cache.kvq_append_decode_attn(0, kn.cuda(), vn.cuda(), q.cuda(), scale=float(scale))
        assert cache.kvq_last_launches() == 2
        lens = [x + 1 for x in lens]
        if s % 13 == 12 or s == steps - 1:
            torch.cuda.synchronize()
            kk = torch.zeros((B, cache.tcap, H, D), dtype=k.dtype)
            vv = torch.zeros_like(kk)
            for i in range(B):
                kk[i, :lens[i]] = k[i, :lens[i]]
                vv[i, :lens[i]] = v[i, :lens[i]]
            ok = oracle_tensor(kk, lens, cache.tcap, kc, False)
            ov = oracle_tensor(vv, lens, cache.tcap, vc, False)
            ref = _rope_ref(wl, ok, ov, lens, q, scale, base)
            assert rel_err_rows(out.cpu().numpy(), ref).max() <= TOL, s
            k16, v16 = cache.kvq_dequantize(0)
            mat = cache.kvq_decode_attn_materialized(0, k16, v16, q.cuda(), scale=float(scale))
            torch.cuda.synchronize()
            assert rel_err_rows(mat.cpu().numpy(), ref).max() <= TOL, s
