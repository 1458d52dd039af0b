"""CPU oracle for group-wise integer KV-cache quantization and decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use this package; the product path
(``bit_quantized_kv_02_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``kvq_oracle.c`` (plain scalar C, built with
``-O2 -ffp-contract=off``: every float operation is one IEEE-754 operation in
source order).  This module only compiles it with gcc and marshals numpy arrays
through ctypes.  Each C function's header comment cites the page section it
follows.

Parity unpinned (conventions the pages leave open, pinned only by invariants
and by the oracle and the CUDA path agreeing): the tie rule, the directed fp16
rounding of the stored zero point and step, and the symmetric code offset.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PER_TOKEN = 0
PER_CHANNEL = 1
WHOLE_VECTOR = -1  # group size meaning "all kv_heads*head_dim channels of a token"

ROUND_NEAREST = 0
ROUND_DOWN = 1
ROUND_UP = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into oracle/_build/libkvq_oracle.so (gcc, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I, L, F = ctypes.c_int, ctypes.c_long, ctypes.c_float
        lib.kvqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.kvqo_f16_to_f32.restype = F
        lib.kvqo_f32_to_f16.argtypes = [F, I]
        lib.kvqo_f32_to_f16.restype = ctypes.c_uint16
        lib.kvqo_f32_to_f16_array.argtypes = [P, L, I, P]
        lib.kvqo_f16_to_f32_array.argtypes = [P, L, P]
        lib.kvqo_quant_group.argtypes = [P, L, L, I, I, I, P, L, P, P]
        lib.kvqo_dequant_one.argtypes = [I, F, F, I, I]
        lib.kvqo_dequant_one.restype = ctypes.c_double
        lib.kvqo_sealed.argtypes = [L, I, I, I]
        lib.kvqo_sealed.restype = L
        lib.kvqo_tail_rows.argtypes = [I, I, I]
        lib.kvqo_tail_rows.restype = L
        lib.kvqo_meta_groups.argtypes = [I, I, I, I, I, I]
        lib.kvqo_meta_groups.restype = L
        lib.kvqo_quantize_tensor.argtypes = [P, I, I, I, I, P, I, I, I, I, I, I, I, P, P, P]
        lib.kvqo_quantize_tensor.restype = I
        lib.kvqo_dequant_tensor.argtypes = [P, P, P, I, I, I, P, I, I, I, I, I, I, P]
        lib.kvqo_dequant_tensor.restype = I
        lib.kvqo_attention.argtypes = [P, P, P, P, I, I, I, I, I, F, P]
        lib.kvqo_attention.restype = I
        lib.kvqo_tensor_bytes.argtypes = [I, I, I, P, I, I, I, I, I, I, P]
        lib.kvqo_rope.argtypes = [P, I, I, I, I, P, ctypes.c_double]
        lib.kvqo_cache_elements.argtypes = [I, ctypes.c_double, I, I]
        lib.kvqo_cache_elements.restype = ctypes.c_double
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ fp16 ----

def f32_to_f16_bits(x, mode: int = ROUND_NEAREST) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().kvqo_f32_to_f16_array(_ptr(x), x.size, mode, _ptr(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().kvqo_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


# ------------------------------------------------------------- quantizer ----

def quant_group(x, bits: int, sym: bool = False, meta_f32: bool = False):
    """Quantize one group.  Returns (codes uint8[n], z, s) with z, s the stored values."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    codes = np.empty(x.size, dtype=np.uint8)
    z = ctypes.c_float()
    s = ctypes.c_float()
    _load().kvqo_quant_group(_ptr(x), x.size, 1, bits, int(sym), int(meta_f32), _ptr(codes), 1,
                             ctypes.byref(z), ctypes.byref(s))
    return codes, np.float32(z.value), np.float32(s.value)


def dequant_one(code: int, z: float, s: float, bits: int, sym: bool = False) -> float:
    return _load().kvqo_dequant_one(int(code), float(z), float(s), bits, int(sym))


def resolve_group(group: int, heads: int, dim: int) -> int:
    return heads * dim if group == WHOLE_VECTOR else group


def sealed(n: int, axis: int, group: int, window: int = 0) -> int:
    """Tokens of a length-n sequence held as codes (the rest stay fp16)."""
    return _load().kvqo_sealed(n, axis, group, window)


def tail_rows(axis: int, group: int, window: int = 0) -> int:
    """fp16 rows per (sequence, head) the unsealed tokens can occupy."""
    return _load().kvqo_tail_rows(axis, group, window)


def meta_groups(batch, heads, dim, tcap, axis, group) -> int:
    return _load().kvqo_meta_groups(batch, heads, dim, tcap, axis, resolve_group(group, heads, dim))


def quantize_tensor(x, lens, tcap: int, bits: int, group: int, axis: int, sym: bool = False,
                    meta_f32: bool = False, window: int = 0):
    """Quantize one layer-tensor.

    x: float array [batch][T][heads][dim] (exact fp32 copies of the source values);
    lens: int [batch]; window: full-precision recent tokens (multiple of 16, 0 = none).
    Returns dict(codes [B][H][tcap][D] uint8, meta [groups][2] f32, tail
    [B][H][tail_rows][D] uint16 fp16 bits of the unsealed tokens (row t - sealed)
    or None when the tensor has no fp16 rows)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    batch, tstride, heads, dim = x.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    g = resolve_group(group, heads, dim)
    codes = np.empty((batch, heads, tcap, dim), dtype=np.uint8)
    meta = np.empty((meta_groups(batch, heads, dim, tcap, axis, g), 2), dtype=np.float32)
    rows = tail_rows(axis, g, window)
    tail = np.zeros((batch, heads, rows, dim), dtype=np.uint16) if rows else None
    rc = _load().kvqo_quantize_tensor(_ptr(x), batch, tstride, heads, dim, _ptr(lens), tcap, bits, g, axis,
                                      int(sym), int(meta_f32), int(window), _ptr(codes), _ptr(meta),
                                      _ptr(tail) if tail is not None else None)
    if rc != 0:
        raise ValueError("oracle: unsupported tensor shape/config")
    return {"codes": codes, "meta": meta, "tail": tail}


def dequant_tensor(q, lens, bits: int, group: int, axis: int, sym: bool = False, window: int = 0) -> np.ndarray:
    """Reconstruct x_hat [B][H][tcap][D] (float64) from quantize_tensor()'s output."""
    codes, meta, tail = q["codes"], q["meta"], q["tail"]
    batch, heads, tcap, dim = codes.shape
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    g = resolve_group(group, heads, dim)
    out = np.empty(codes.shape, dtype=np.float64)
    rc = _load().kvqo_dequant_tensor(_ptr(np.ascontiguousarray(codes)), _ptr(np.ascontiguousarray(meta)),
                                     _ptr(np.ascontiguousarray(tail)) if tail is not None else None,
                                     batch, heads, dim, _ptr(lens), tcap, bits, g, axis, int(sym), int(window),
                                     _ptr(out))
    if rc != 0:
        raise ValueError("oracle: dequant failed (missing tail?)")
    return out


def attention(khat, vhat, q, lens, scale: float) -> np.ndarray:
    """fp64 single-token decode attention.  khat, vhat: [B][Hkv][T][D] float64;
    q: [B][Hq][D] (fp32 values); returns out [B][Hq][D] float64."""
    khat = np.ascontiguousarray(khat, dtype=np.float64)
    vhat = np.ascontiguousarray(vhat, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    batch, kvh, tcap, dim = khat.shape
    qh = q.shape[1]
    out = np.empty((batch, qh, dim), dtype=np.float64)
    rc = _load().kvqo_attention(_ptr(khat), _ptr(vhat), _ptr(q), _ptr(lens), batch, qh, kvh, dim, tcap,
                                float(np.float32(scale)), _ptr(out))
    if rc != 0:
        raise ValueError("oracle: bad head counts")
    return out


def rope(x, lens, base: float) -> np.ndarray:
    """Rotary position embedding of [B][H][T][D] float64 rows (row t = the token
    at position t), rows t < lens[b]; returns a rotated copy."""
    x = np.array(x, dtype=np.float64, order="C", copy=True)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    batch, heads, tcap, dim = x.shape
    _load().kvqo_rope(_ptr(x), batch, heads, dim, tcap, _ptr(lens), float(base))
    return x


def tensor_bytes(batch, heads, dim, lens, bits, group, axis, sym=False, meta_f32=False, window=0):
    """(packed, metadata, tail) bytes of one layer-tensor holding lens tokens."""
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros(3, dtype=np.float64)
    _load().kvqo_tensor_bytes(batch, heads, dim, _ptr(lens), bits, resolve_group(group, heads, dim), axis,
                              int(sym), int(meta_f32), int(window), _ptr(out))
    return tuple(float(v) for v in out)


def cache_elements(layers: int, tokens: float, kv_heads: int, dim: int) -> float:
    return _load().kvqo_cache_elements(layers, float(tokens), kv_heads, dim)
