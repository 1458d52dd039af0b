"""Pins for the oracle's decode attention and size arithmetic.

Attention is the plain softmax(q.k * scale) . v definition ("Kuantisasi KV
Cache untuk Mengurangi Memory Inferensi Long Context", section "Key dan value
dapat memiliki struktur numerik berbeda": keys enter a dot product with the
current query before the softmax, values are combined with the resulting
weights).  Pinned against torch's scaled_dot_product_attention in fp64 (a
library routine the oracle does not call) and closed forms.

Sizes: section "Ukuran cache bertambah mengikuti token, layer, dan KV head"
(elements = 2*layers*tokens*kv_heads*head_dim) and the ratios printed in
"Asymetrie kvantizace KV cache".
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_attention_matches_torch_sdpa_fp64():
    B, Hq, Hkv, T, D = 2, 8, 2, 37, 64
    k = _rand((B, Hkv, T, D), 1)
    v = _rand((B, Hkv, T, D), 2)
    q = _rand((B, Hq, D), 3).astype(np.float32)
    lens = np.array([37, 20], np.int32)
    scale = np.float32(1.0 / np.sqrt(D))
    out = oracle.attention(k, v, q, lens, scale)
    rep = Hq // Hkv
    for b in range(B):
        n = lens[b]
        kk = torch.from_numpy(np.repeat(k[b, :, :n], rep, axis=0))  # [Hq][n][D]
        vv = torch.from_numpy(np.repeat(v[b, :, :n], rep, axis=0))
        qq = torch.from_numpy(q[b].astype(np.float64))[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=float(scale))[:, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    B, H, T, D = 1, 1, 9, 8
    k = _rand((B, H, T, D), 4)
    v = _rand((B, H, T, D), 5)
    q = _rand((B, H, D), 6).astype(np.float32)
    s = np.float32(0.3)
    # one token: the output is that token's value
    out = oracle.attention(k, v, q, np.array([1], np.int32), s)
    np.testing.assert_array_equal(out[0, 0], v[0, 0, 0])
    # constant values: the output is that constant
    vc = np.broadcast_to(v[:, :, :1, :], v.shape).copy()
    out = oracle.attention(k, vc, q, np.array([T], np.int32), s)
    np.testing.assert_allclose(out[0, 0], v[0, 0, 0], rtol=1e-14)
    # zero query: uniform weights, the output is the mean value
    out = oracle.attention(k, v, np.zeros_like(q), np.array([T], np.int32), s)
    np.testing.assert_allclose(out[0, 0], v[0, 0].mean(axis=0), rtol=1e-13)
    # adding one vector to every key shifts all scores equally: output unchanged
    out1 = oracle.attention(k, v, q, np.array([T], np.int32), s)
    out2 = oracle.attention(k + _rand((1, 1, 1, D), 7), v, q, np.array([T], np.int32), s)
    np.testing.assert_allclose(out1, out2, rtol=1e-12, atol=1e-13)
    # empty sequence: zeros
    out = oracle.attention(k, v, q, np.array([0], np.int32), s)
    assert not out.any()


def test_gqa_head_mapping_consecutive():
    B, Hq, Hkv, T, D = 1, 6, 3, 5, 4
    k = _rand((B, Hkv, T, D), 8)
    v = _rand((B, Hkv, T, D), 9)
    q = np.repeat(_rand((B, 1, D), 10), Hq, axis=1).astype(np.float32)
    out = oracle.attention(k, v, q, np.array([T], np.int32), np.float32(0.5))
    # query heads 2j, 2j+1 share kv head j; different kv heads differ
    for j in range(Hkv):
        np.testing.assert_array_equal(out[0, 2 * j], out[0, 2 * j + 1])
        single = oracle.attention(k[:, j:j + 1], v[:, j:j + 1], q[:, :1], np.array([T], np.int32), np.float32(0.5))
        np.testing.assert_array_equal(out[0, 2 * j], single[0, 0])
    assert not np.allclose(out[0, 0], out[0, 2])


def test_attention_oracle_over_dequantized_cache():
    """End-to-end oracle: quantize, dequantize, attend; close to full precision at 8 bits."""
    rng = np.random.default_rng(11)
    B, T, H, D = 1, 96, 2, 64
    k = rng.standard_normal((B, T, H, D)).astype(np.float32)
    v = rng.standard_normal((B, T, H, D)).astype(np.float32)
    q = rng.standard_normal((B, H, D)).astype(np.float32)
    lens = np.array([T], np.int32)
    qk = oracle.quantize_tensor(k, lens, T, 8, 32, oracle.PER_CHANNEL)
    qv = oracle.quantize_tensor(v, lens, T, 8, 32, oracle.PER_TOKEN)
    kh = oracle.dequant_tensor(qk, lens, 8, 32, oracle.PER_CHANNEL)
    vh = oracle.dequant_tensor(qv, lens, 8, 32, oracle.PER_TOKEN)
    s = np.float32(1 / 8)
    o_q = oracle.attention(kh, vh, q, lens, s)
    o_f = oracle.attention(k.transpose(0, 2, 1, 3), v.transpose(0, 2, 1, 3), q, lens, s)
    assert np.max(np.abs(o_q - o_f)) < 0.02


# ------------------------------------------------------------------ sizes ----

def test_element_count_closed_form():
    assert oracle.cache_elements(40, 4096, 40, 128) == 2 * 40 * 4096 * 40 * 128
    assert oracle.cache_elements(12, 2048, 12, 64) == 2 * 12 * 2048 * 12 * 64


def _effective_bits(H, D, kbits, vbits, kgroup, vgroup, kaxis, vaxis, T=4096):
    lens = np.array([T], np.int32)
    pk, mk, tk = oracle.tensor_bytes(1, H, D, lens, kbits, kgroup, kaxis)
    pv, mv, tv = oracle.tensor_bytes(1, H, D, lens, vbits, vgroup, vaxis)
    elems = 2 * T * H * D
    return 8 * (pk + mk + tk + pv + mv + tv) / elems


def test_gpt2_k6v4_effective_bits_and_ratio():
    g = GOLD["gpt2_small"]
    H, D, G = g["shape"]["kv_heads"], g["shape"]["head_dim"], g["per_head_group_channels"]
    eb = _effective_bits(H, D, 6, 4, G, G, oracle.PER_TOKEN, oracle.PER_TOKEN)
    assert eb == pytest.approx(g["k6v4_effective_bits"], abs=1e-12)
    assert round(16 / eb, 1) == g["k6v4_size_ratio_printed"]
    # the knee: 5.5 .. 6.5 effective bits <-> 2.9x .. 2.5x smaller than fp16
    lo, hi = g["knee_effective_bits"]
    eb_hi = _effective_bits(H, D, 6, 6, G, G, oracle.PER_TOKEN, oracle.PER_TOKEN)
    assert eb_hi == pytest.approx(hi)
    assert [round(16 / hi, 1), round(16 / lo, 1)] == g["knee_size_ratio_printed"]


def test_hybrid_model_k4v8_ratio_and_saving():
    g = GOLD["hybrid_model"]
    L, D, T, H = g["full_attention_layers"], g["head_dim"], g["context_tokens"], g["kv_heads_reading"]
    fp16_bytes = 2 * oracle.cache_elements(L, T, H, D)
    assert round(fp16_bytes / 1e9, 1) == g["bf16_cache_gb_printed"]
    eb = _effective_bits(H, D, 4, 8, D, D, oracle.PER_TOKEN, oracle.PER_TOKEN, T=T)
    assert eb == pytest.approx(6.125)
    assert round(16 / eb, 1) == g["k4v8_size_ratio_printed"]
    saved = fp16_bytes * (1 - eb / 16)
    assert round(saved / 1e9, 1) == g["k4v8_saved_gb_printed"]


def test_tail_counts_two_bytes_per_element():
    lens = np.array([4113], np.int32)  # 4096 sealed + 17 tail tokens
    p, m, t = oracle.tensor_bytes(1, 40, 128, lens, 2, 32, oracle.PER_CHANNEL)
    assert t == 17 * 40 * 128 * 2
    assert p == 4096 * 40 * 128 * 2 / 8
    assert m == (4096 // 32) * 40 * 128 * 4
