"""Quantization-axis study (the pages' orderings on synthetic outlier data).

"O Seu Cache KV Nao Tem um Problema de Bits. Tem um Problema de Geometria",
sections "Chaves: Os Valores Extremos Vivem em Canais Fixos" and "Valores: Onde
a Intuicao Quebra": with fixed outlier key channels, keys grouped per channel
have lower error than keys grouped per token; for values the stored-tensor
error favours (slightly) per-channel groups while the attention-output error,
under sparse attention, is several times lower with per-token groups.  The CPU
tests compute the study with the oracle; the GPU test repeats it through the
C ABI (kvq_dequantize rows and kvq_decode_attn outputs).
"""
import numpy as np
import pytest
import torch

from bit_quantized_kv_02_gb300 import synth
from tests import axis_study


@pytest.fixture(scope="module")
def study():
    return {b: axis_study.run(bits=b) for b in (2, 4)}


def _row(res, ka, va):
    return next(r for r in res["rows"] if r["keys"] == ka and r["values"] == va)


def test_attention_is_sparse(study):
    # the page reports 84.3 % attention sparsity; the inputs aim at that regime
    assert 0.8 <= study[2]["important_mass"] <= 0.9


@pytest.mark.parametrize("bits", [2, 4])
def test_keys_per_channel_beat_per_token(study, bits):
    res = study[bits]
    pc, pt = _row(res, "per-channel", "per-token"), _row(res, "per-token", "per-token")
    assert pc["key_error"] < 0.8 * pt["key_error"]
    assert pc["logit_error"] < 0.6 * pt["logit_error"]


@pytest.mark.parametrize("bits", [2, 4])
def test_values_stored_error_and_output_error_disagree(study, bits):
    res = study[bits]
    pt, pc = _row(res, "per-channel", "per-token"), _row(res, "per-channel", "per-channel")
    # the stored tensor favours per-channel values...
    assert pc["value_error"] < pt["value_error"]
    # ...the attention output favours per-token values by a wide margin
    assert pt["output_error"] * 3.0 < pc["output_error"]


@pytest.mark.gpu
def test_study_through_the_cuda_path():
    """The same orderings with the GPU quantizer (kvq_dequantize rows) and the
    GPU decode attention (kvq_decode_attn) in place of the oracle."""
    from bit_quantized_kv_02_gb300 import build, kvq
    build.build()
    k, v, q, _ = synth.axis_study_inputs()
    T, H, D = k.shape[1], k.shape[2], k.shape[3]
    scale = float(np.float32(1.0 / np.sqrt(D)))
    k64 = k[0].permute(1, 0, 2).double()  # [H][T][D]
    v64 = v[0].permute(1, 0, 2).double()
    q64 = q[0].double()
    p = torch.softmax(torch.einsum("hd,htd->ht", q64, k64) * scale, dim=-1)
    out_ref = torch.einsum("ht,htd->hd", p, v64)
    err = {}
    for ka, va in axis_study.COMBOS:
        tk = (2, 32, kvq.PER_CHANNEL if ka == "per-channel" else kvq.PER_TOKEN, kvq.ASYM)
        tv = (2, 32, kvq.PER_CHANNEL if va == "per-channel" else kvq.PER_TOKEN, kvq.ASYM)
        cache = kvq.KVQCache(kvq.make_config(1, 1, H, H, D, T, tk, tv))
        cache.kvq_prefill_quantize(0, k.cuda(), v.cuda(), [T])
        k16, v16 = cache.kvq_dequantize(0)
        out = cache.kvq_decode_attn(0, q.cuda().float(), scale=scale)
        torch.cuda.synchronize()
        kh = k16[0].double().cpu()
        vh = v16[0].double().cpu()
        err[(ka, va)] = {"key": float((kh - k64).norm() / k64.norm()), "value": float((vh - v64).norm() / v64.norm()),
                         "output": float((out[0].double().cpu() - out_ref).norm() / out_ref.norm())}
    assert err[("per-channel", "per-token")]["key"] < 0.8 * err[("per-token", "per-token")]["key"]
    assert err[("per-channel", "per-channel")]["value"] < err[("per-channel", "per-token")]["value"]
    assert err[("per-channel", "per-token")]["output"] * 3.0 < err[("per-channel", "per-channel")]["output"]
