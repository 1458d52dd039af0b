"""Quantization-axis study on synthetic outlier data, computed with the oracle.

Restates, on seeded synthetic inputs, the orderings of "O Seu Cache KV Nao Tem
um Problema de Bits. Tem um Problema de Geometria": section "Chaves: Os Valores
Extremos Vivem em Canais Fixos" (keys grouped per channel beat keys grouped per
token when outliers sit in fixed channels) and section "Valores: Onde a
Intuicao Quebra" (for values, the reconstruction error of the stored tensor
barely separates the two axes or even favours per-channel groups, while the
error of the attention output, under sparse attention, is far lower for
per-token groups).  The numbers are this data's, not the page's.

Run `python -m tests.axis_study` for the table.  Test infrastructure: it uses
the oracle and only the test suite imports it.
"""
from __future__ import annotations

import numpy as np

import oracle
from bit_quantized_kv_02_gb300 import synth

COMBOS = [("per-channel", "per-token"), ("per-channel", "per-channel"), ("per-token", "per-token"),
          ("per-token", "per-channel")]
AXIS = {"per-token": oracle.PER_TOKEN, "per-channel": oracle.PER_CHANNEL}


def _dequant(x, bits, group, axis):
    T = x.shape[1]
    lens = np.array([T], np.int32)
    q = oracle.quantize_tensor(x, lens, T, bits, group, axis)
    return oracle.dequant_tensor(q, lens, bits, group, axis)  # [1][H][T][D]


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def run(bits=2, group=32, seed=0, **inputs):
    """Errors of every (key axis, value axis) combination: relative Frobenius
    error of the stored keys and values, of the attention logits q.k/sqrt(D),
    and of the attention output, each against the unquantized fp64 values."""
    k, v, q, imp = synth.axis_study_inputs(seed=seed, **inputs)
    kx = k.numpy().astype(np.float32)
    vx = v.numpy().astype(np.float32)
    qx = q.numpy().astype(np.float32)
    T, H, D = kx.shape[1], kx.shape[2], kx.shape[3]
    lens = np.array([T], np.int32)
    scale = np.float32(1.0 / np.sqrt(D))
    k_ref = kx.transpose(0, 2, 1, 3).astype(np.float64)  # [1][H][T][D]
    v_ref = vx.transpose(0, 2, 1, 3).astype(np.float64)
    logits_ref = np.einsum("bhd,bhtd->bht", qx.astype(np.float64), k_ref) * float(scale)
    out_ref = oracle.attention(k_ref, v_ref, qx, lens, scale)
    p = np.exp(logits_ref - logits_ref.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    sparsity = float(p[..., imp.numpy()].sum(axis=-1).mean())
    kh = {a: _dequant(kx, bits, group, AXIS[a]) for a in AXIS}
    vh = {a: _dequant(vx, bits, group, AXIS[a]) for a in AXIS}
    rows = []
    for ka, va in COMBOS:
        logits = np.einsum("bhd,bhtd->bht", qx.astype(np.float64), kh[ka]) * float(scale)
        out = oracle.attention(kh[ka], vh[va], qx, lens, scale)
        rows.append({"keys": ka, "values": va, "key_error": _rel(kh[ka], k_ref), "value_error": _rel(vh[va], v_ref),
                     "logit_error": _rel(logits, logits_ref), "output_error": _rel(out, out_ref)})
    return {"bits": bits, "group": group, "tokens": T, "heads": H, "head_dim": D,
            "important_mass": sparsity, "rows": rows}


def table(res) -> str:
    lines = [f"{res['bits']}-bit, groups of {res['group']}, {res['tokens']} tokens x {res['heads']} heads x "
             f"{res['head_dim']}; softmax mass on the important tokens: {res['important_mass']:.3f}",
             "| keys | values | key error | value error | logit error | output error |", "|---|---|---|---|---|---|"]
    for r in res["rows"]:
        lines.append(f"| {r['keys']} | {r['values']} | {r['key_error']:.4f} | {r['value_error']:.4f} | "
                     f"{r['logit_error']:.4f} | {r['output_error']:.4f} |")
    return "\n".join(lines)


if __name__ == "__main__":
    for b in (2, 4):
        print(table(run(bits=b)))
        print()
