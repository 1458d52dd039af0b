"""Thin ctypes binding of libkvq (include/kvq.h): argument marshalling only.

Every step of the quantize / append / decode path runs in the CUDA kernels of
libkvq.so; PyTorch only provides device memory and the CUDA stream.  There is
no CPU fallback: if the library is missing the calls raise.

The functions keep the C names (``kvq_cache_bytes``, ``kvq_cache_create``,
``kvq_prefill_quantize``, ``kvq_append``, ``kvq_decode_attn``, ``kvq_export``,
...); ``KVQCache`` wraps a handle plus the torch buffer it lives in.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PER_TOKEN, PER_CHANNEL = 0, 1
ASYM, SYM = 0, 1
F16, F32 = 0, 1
WHOLE_VECTOR = -1

STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CAPACITY",
          4: "KVQ_ERR_BUFFER_TOO_SMALL", 5: "KVQ_ERR_CUDA", 6: "KVQ_ERR_DEVICE_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")


class KVQError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class TensorCfg(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int), ("group", ctypes.c_int), ("axis", ctypes.c_int), ("mode", ctypes.c_int)]


class Config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("batch", ctypes.c_int), ("q_heads", ctypes.c_int),
                ("kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("k", TensorCfg), ("v", TensorCfg), ("meta_dtype", ctypes.c_int), ("max_splits", ctypes.c_int),
                ("recent_window", ctypes.c_int), ("rope_theta", ctypes.c_float)]


class Bytes(ctypes.Structure):
    _fields_ = [("tail", ctypes.c_double), ("packed", ctypes.c_double), ("metadata", ctypes.c_double),
                ("workspace", ctypes.c_double), ("total", ctypes.c_double), ("elements", ctypes.c_double),
                ("alloc", ctypes.c_size_t)]


_lock = threading.Lock()
_lib = None

EXPORTED = ["kvq_cache_bytes", "kvq_cache_create", "kvq_cache_destroy", "kvq_prefill_quantize", "kvq_append",
            "kvq_decode_attn", "kvq_export", "kvq_cache_tcap", "kvq_get_lens", "kvq_decode_traffic",
            "kvq_device_status", "kvq_last_launches", "kvq_status_string", "kvq_last_error",
            "kvq_set_decode_plan", "kvq_refresh_lens", "kvq_decode_attn_static", "kvq_set_decode_kernel",
            "kvq_decode_kernel_specialized", "kvq_dequantize", "kvq_decode_attn_materialized",
            "kvq_append_decode_attn", "kvq_decode_cta_warps"]


def lib():
    """Load libkvq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkvq.so not built ({LIB_PATH}); run bit_quantized_kv_02_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        L.kvq_cache_bytes.argtypes = [ctypes.POINTER(Config), P, ctypes.POINTER(Bytes)]
        L.kvq_cache_create.argtypes = [ctypes.POINTER(Config), P, ctypes.c_size_t, P, ctypes.POINTER(P)]
        L.kvq_cache_destroy.argtypes = [P]
        L.kvq_prefill_quantize.argtypes = [P, I, P, P, I, P, ctypes.c_int64, P]
        L.kvq_append.argtypes = [P, I, P, P, I, P]
        L.kvq_decode_attn.argtypes = [P, I, P, I, ctypes.c_float, P, P]
        L.kvq_append_decode_attn.argtypes = [P, I, P, P, I, P, I, ctypes.c_float, P, P]
        L.kvq_export.argtypes = [P, I, P, P, P, P, P, P, P, P]
        L.kvq_cache_tcap.argtypes = [P]
        L.kvq_cache_tcap.restype = I
        L.kvq_get_lens.argtypes = [P, I, P]
        L.kvq_decode_traffic.argtypes = [P, I, I, ctypes.POINTER(ctypes.c_double)]
        L.kvq_device_status.argtypes = [P, P]
        L.kvq_last_launches.argtypes = [P]
        L.kvq_last_launches.restype = I
        L.kvq_status_string.argtypes = [S]
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_decode_attn_static.argtypes = [P, I, P, I, ctypes.c_float, P, P]
        L.kvq_dequantize.argtypes = [P, I, P, P, P]
        L.kvq_decode_attn_materialized.argtypes = [P, I, P, P, P, I, ctypes.c_float, P, P]
        L.kvq_set_decode_plan.argtypes = [P, I]
        L.kvq_set_decode_kernel.argtypes = [P, I]
        L.kvq_decode_kernel_specialized.argtypes = [P]
        L.kvq_decode_kernel_specialized.restype = I
        L.kvq_decode_cta_warps.argtypes = [P, I]
        L.kvq_decode_cta_warps.restype = I
        L.kvq_refresh_lens.argtypes = [P, P]
        L.kvq_last_error.argtypes = [P]
        L.kvq_last_error.restype = ctypes.c_char_p
        for name in ("kvq_cache_bytes", "kvq_cache_create", "kvq_cache_destroy", "kvq_prefill_quantize",
                     "kvq_append", "kvq_decode_attn", "kvq_export", "kvq_get_lens", "kvq_decode_traffic",
                     "kvq_device_status", "kvq_set_decode_plan", "kvq_refresh_lens", "kvq_decode_attn_static",
                     "kvq_set_decode_kernel", "kvq_dequantize", "kvq_decode_attn_materialized"):
            getattr(L, name).restype = S
        _lib = L
        return L


def make_config(layers, batch, q_heads, kv_heads, head_dim, max_tokens, k, v, meta_dtype=F16, max_splits=0,
                recent_window=0, rope_theta=0.0):
    """k, v: (bits, group, axis, mode) tuples or dicts; recent_window: fp16 window
    of the newest tokens of both tensors (multiple of 16, 0 = none); rope_theta:
    base of the rotary embedding applied to the dequantized keys at decode (keys
    cached before RoPE; 0 = none)."""
    def tc(t):
        if isinstance(t, dict):
            return TensorCfg(t["bits"], t["group"], t["axis"], t.get("mode", ASYM))
        return TensorCfg(*t)
    return Config(layers, batch, q_heads, kv_heads, head_dim, max_tokens, tc(k), tc(v), meta_dtype, max_splits,
                  recent_window, float(rope_theta))


def _check(st: int, what: str, handle=None):
    if st != 0:
        detail = ""
        if handle is not None:
            detail = (lib().kvq_last_error(handle) or b"").decode()
        raise KVQError(st, what, detail)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (fp16 or fp32)")


# ------------------------------------------------------- C-named functions --

def kvq_cache_bytes(cfg: Config, lens=None) -> Bytes:
    out = Bytes()
    arr = None
    if lens is not None:
        arr = (ctypes.c_int32 * len(lens))(*[int(x) for x in lens])
    _check(lib().kvq_cache_bytes(ctypes.byref(cfg), arr, ctypes.byref(out)), "kvq_cache_bytes")
    return out


def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(status).decode()


class KVQCache:
    """A libkvq cache handle living in one torch uint8 device buffer."""

    def __init__(self, cfg: Config, device="cuda", stream=None):
        self.cfg = cfg
        self.bytes = kvq_cache_bytes(cfg)
        self.buffer = torch.empty(self.bytes.alloc, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        _check(lib().kvq_cache_create(ctypes.byref(cfg), _ptr(self.buffer), self.bytes.alloc, _stream(stream),
                                      ctypes.byref(h)), "kvq_cache_create")
        self.handle = h
        self.tcap = lib().kvq_cache_tcap(h)

    def close(self):
        if getattr(self, "handle", None):
            lib().kvq_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # C-named methods ---------------------------------------------------------
    def kvq_prefill_quantize(self, layer: int, k: torch.Tensor, v: torch.Tensor, lens, stream=None):
        """k, v: [batch][T][kv_heads][head_dim] contiguous fp16/fp32 on the device."""
        assert k.is_contiguous() and v.is_contiguous() and k.shape == v.shape and k.dtype == v.dtype
        arr = (ctypes.c_int32 * self.cfg.batch)(*[int(x) for x in lens])
        _check(lib().kvq_prefill_quantize(self.handle, layer, _ptr(k), _ptr(v), _dtype_code(k), arr, k.shape[1],
                                          _stream(stream)), "kvq_prefill_quantize", self.handle)

    def kvq_append(self, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """k_new, v_new: [batch][kv_heads][head_dim] contiguous fp16/fp32 on the device."""
        assert k_new.is_contiguous() and v_new.is_contiguous() and k_new.dtype == v_new.dtype
        _check(lib().kvq_append(self.handle, layer, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _stream(stream)),
               "kvq_append", self.handle)

    def kvq_decode_attn(self, layer: int, q: torch.Tensor, out: torch.Tensor | None = None, scale: float = 0.0,
                        stream=None) -> torch.Tensor:
        """q: [batch][q_heads][head_dim] fp16/fp32; returns fp32 [batch][q_heads][head_dim]."""
        assert q.is_contiguous()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _check(lib().kvq_decode_attn(self.handle, layer, _ptr(q), _dtype_code(q), float(scale), _ptr(out),
                                     _stream(stream)), "kvq_decode_attn", self.handle)
        return out

    def kvq_append_decode_attn(self, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                               out: torch.Tensor | None = None, scale: float = 0.0, stream=None) -> torch.Tensor:
        """kvq_append then kvq_decode_attn on `layer`, in one launch where the
        layout allows it: k_new, v_new [batch][kv_heads][head_dim]; q
        [batch][q_heads][head_dim]; returns fp32 [batch][q_heads][head_dim]."""
        assert k_new.is_contiguous() and v_new.is_contiguous() and k_new.dtype == v_new.dtype
        assert q.is_contiguous()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _check(lib().kvq_append_decode_attn(self.handle, layer, _ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                                            _ptr(q), _dtype_code(q), float(scale), _ptr(out), _stream(stream)),
               "kvq_append_decode_attn", self.handle)
        return out

    def kvq_decode_attn_static(self, layer: int, q: torch.Tensor, out: torch.Tensor | None = None,
                               scale: float = 0.0, stream=None) -> torch.Tensor:
        """kvq_decode_attn with its scratch in the library's static device array
        (for callers that cannot provide device memory); same inputs and output."""
        assert q.is_contiguous()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _check(lib().kvq_decode_attn_static(self.handle, layer, _ptr(q), _dtype_code(q), float(scale), _ptr(out),
                                            _stream(stream)), "kvq_decode_attn_static", self.handle)
        return out

    def kvq_dequantize(self, layer: int, k_out: torch.Tensor | None = None, v_out: torch.Tensor | None = None,
                       stream=None):
        """Materialised baseline: fp16 K and V rows [batch][kv_heads][tcap][head_dim]
        of `layer` (rows past a sequence's length are left as they were)."""
        c = self.cfg
        shape = (c.batch, c.kv_heads, self.tcap, c.head_dim)
        if k_out is None:
            k_out = torch.zeros(shape, dtype=torch.float16, device=self.buffer.device)
        if v_out is None:
            v_out = torch.zeros(shape, dtype=torch.float16, device=self.buffer.device)
        assert k_out.shape == shape and v_out.shape == shape and k_out.dtype == torch.float16
        assert k_out.is_contiguous() and v_out.is_contiguous() and v_out.dtype == torch.float16
        _check(lib().kvq_dequantize(self.handle, layer, _ptr(k_out), _ptr(v_out), _stream(stream)), "kvq_dequantize",
               self.handle)
        return k_out, v_out

    def kvq_decode_attn_materialized(self, layer: int, k16: torch.Tensor, v16: torch.Tensor, q: torch.Tensor,
                                     out: torch.Tensor | None = None, scale: float = 0.0,
                                     stream=None) -> torch.Tensor:
        """Decode attention over rows from kvq_dequantize (the baseline the fused
        kvq_decode_attn is measured against); same query and output layout."""
        assert q.is_contiguous() and k16.is_contiguous() and v16.is_contiguous()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        _check(lib().kvq_decode_attn_materialized(self.handle, layer, _ptr(k16), _ptr(v16), _ptr(q), _dtype_code(q),
                                                  float(scale), _ptr(out), _stream(stream)),
               "kvq_decode_attn_materialized", self.handle)
        return out

    def kvq_export(self, layer: int, stream=None) -> dict:
        c = self.cfg
        dev = self.buffer.device
        B, H, D, T = c.batch, c.kv_heads, c.head_dim, self.tcap

        def groups(t):
            if t.axis == PER_CHANNEL:
                return B * H * (T // t.group) * D
            if t.group == WHOLE_VECTOR:
                return B * T
            return B * H * T * (D // t.group)

        def rows(t):  # fp16 rows per (sequence, head): the unsealed tokens, row t - sealed
            if t.axis == PER_CHANNEL:
                return t.group + c.recent_window
            return c.recent_window + 16 if c.recent_window else 0

        out = {
            "codes_k": torch.zeros((B, H, T, D), dtype=torch.uint8, device=dev),
            "codes_v": torch.zeros((B, H, T, D), dtype=torch.uint8, device=dev),
            "meta_k": torch.zeros((groups(c.k), 2), dtype=torch.float32, device=dev),
            "meta_v": torch.zeros((groups(c.v), 2), dtype=torch.float32, device=dev),
            "tail_k": torch.zeros((B, H, rows(c.k), D), dtype=torch.int16, device=dev) if rows(c.k) else None,
            "tail_v": torch.zeros((B, H, rows(c.v), D), dtype=torch.int16, device=dev) if rows(c.v) else None,
            "lens": torch.zeros((B,), dtype=torch.int32, device=dev),
        }
        _check(lib().kvq_export(self.handle, layer, _ptr(out["codes_k"]), _ptr(out["codes_v"]), _ptr(out["meta_k"]),
                                _ptr(out["meta_v"]), _ptr(out["tail_k"]), _ptr(out["tail_v"]), _ptr(out["lens"]),
                                _stream(stream)), "kvq_export", self.handle)
        return out

    def kvq_get_lens(self, layer: int):
        arr = (ctypes.c_int32 * self.cfg.batch)()
        _check(lib().kvq_get_lens(self.handle, layer, arr), "kvq_get_lens", self.handle)
        return list(arr)

    def kvq_decode_traffic(self, layer: int, q_dtype: int = F16) -> float:
        v = ctypes.c_double()
        _check(lib().kvq_decode_traffic(self.handle, layer, q_dtype, ctypes.byref(v)), "kvq_decode_traffic")
        return v.value

    def kvq_device_status(self, stream=None) -> int:
        return lib().kvq_device_status(self.handle, _stream(stream))

    def kvq_set_decode_plan(self, plan_tokens: int):
        _check(lib().kvq_set_decode_plan(self.handle, int(plan_tokens)), "kvq_set_decode_plan")

    def kvq_set_decode_kernel(self, which: int):
        """0: compile-time specialisation when one matches (default); 1: generic kernel."""
        _check(lib().kvq_set_decode_kernel(self.handle, int(which)), "kvq_set_decode_kernel", self.handle)

    def kvq_decode_cta_warps(self, fused: bool = False) -> int:
        """Warps per CTA of the current decode (fused: decode-step) kernel; 0 if the step runs two kernels."""
        return int(lib().kvq_decode_cta_warps(self.handle, int(bool(fused))))

    def kvq_decode_kernel_specialized(self) -> bool:
        return bool(lib().kvq_decode_kernel_specialized(self.handle))

    def kvq_refresh_lens(self, stream=None):
        _check(lib().kvq_refresh_lens(self.handle, _stream(stream)), "kvq_refresh_lens", self.handle)

    def kvq_last_launches(self) -> int:
        return lib().kvq_last_launches(self.handle)
