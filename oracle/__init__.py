"""CPU oracle for paged decode attention and the slot-mapped KV append.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg (and its ``--impl reference`` arm) may
import this package.  The product library never imports, links or calls it,
and this package never imports the product library: the two share no code.
The only module both sides use is the seeded input generator, which holds
none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, its own binary16
decode and round-to-nearest-even encode).  This module compiles it with gcc
and marshals numpy arrays to it with ctypes; it computes nothing itself.

What each function follows (page title, section):
  * ``decode``  -- "Distributed LLM Inference Serving Platform", sections 2,
    3 and 5.1: gather each sequence's tokens in logical order through its
    block table, softmax(q K^T * scale) V per query head, query head h reading
    KV head h / (n_q_heads / n_kv_heads).
  * ``append``  -- same page, section 5.1: the new token's K/V vectors are
    written into their assigned physical block slot.
  * ``partial`` / ``lse_merge`` -- the log-sum-exp split of the same softmax
    (FlashAttention-2, cited in section 14 of that page).
  * ``decode_multi`` -- several new tokens per sequence attending causally
    over the paged cache (speculative-decoding verify and chunked prefill:
    the roadmap page's Deferred list, and section 9.2 of the serving page).
  * ``e4m3_*``, ``append_f8``, ``decode_f8`` -- the FP8 KV cache that
    "Roadmap: vLLM-style serving features for TornadoVM batched decode" (KV
    cache list) names as future work; the format (OCP E4M3, per-tensor
    scales, round-to-nearest-even with saturation) is this library's reading.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (OpenMP on)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    c = ctypes
    p = c.c_void_p
    lib.pkvo_f16_to_f64.argtypes = [c.c_uint16]
    lib.pkvo_f16_to_f64.restype = c.c_double
    lib.pkvo_f64_to_f16.argtypes = [c.c_double]
    lib.pkvo_f64_to_f16.restype = c.c_uint16
    lib.pkvo_init.argtypes = []
    lib.pkvo_init.restype = None
    lib.pkvo_append.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64]
    lib.pkvo_append.restype = c.c_int
    lib.pkvo_decode.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_double,
                                c.c_int, c.c_int, c.c_int, c.c_int, p, p, p, p, c.c_int]
    lib.pkvo_decode.restype = c.c_int
    lib.pkvo_decode_partial.argtypes = [p, p, p, p, c.c_int, c.c_int64, c.c_double, c.c_int,
                                        c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                        c.c_int, p, p, p]
    lib.pkvo_decode_partial.restype = c.c_int
    lib.pkvo_lse_merge.argtypes = [c.c_int, p, p, p, c.c_int, p, p]
    lib.pkvo_lse_merge.restype = None
    lib.pkvo_e4m3_to_f64.argtypes = [c.c_uint8]
    lib.pkvo_e4m3_to_f64.restype = c.c_double
    lib.pkvo_f32_to_e4m3.argtypes = [c.c_float]
    lib.pkvo_f32_to_e4m3.restype = c.c_uint8
    lib.pkvo_quantize_e4m3_array.argtypes = [p, c.c_int64, c.c_float, p]
    lib.pkvo_quantize_e4m3_array.restype = None
    lib.pkvo_f32_to_e4m3_array.argtypes = [p, c.c_int64, p]
    lib.pkvo_f32_to_e4m3_array.restype = None
    lib.pkvo_append_f8.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64,
                                   c.c_float, c.c_float]
    lib.pkvo_append_f8.restype = c.c_int
    lib.pkvo_decode_f8.argtypes = [p, p, p, c.c_double, c.c_double, p, p, c.c_int, c.c_int,
                                   c.c_int64, c.c_double, c.c_int, c.c_int, c.c_int, c.c_int, p,
                                   p, p, c.c_int]
    lib.pkvo_decode_f8.restype = c.c_int
    lib.pkvo_decode_multi.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_double,
                                      c.c_int, c.c_int, c.c_int, c.c_int, p, p, c.c_int]
    lib.pkvo_decode_multi.restype = c.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
            _lib.pkvo_init()
        return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _u16(a):
    """View an fp16 (or uint16) array as contiguous uint16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16/uint16 bits, got {a.dtype}")
    return a


class OracleError(ValueError):
    """The oracle rejected its input (bad block id, context length or heads)."""


def f16_to_f64(bits: int, lib=None) -> float:
    return (lib or load()).pkvo_f16_to_f64(int(bits))


def f64_to_f16(x: float, lib=None) -> int:
    return int((lib or load()).pkvo_f64_to_f16(float(x)))


def append(k_new, v_new, slot_mapping, k_cache, v_cache, block_size, lib=None):
    """Slot-mapped append into copies of the caches.

    k_new, v_new: [T, Hk, d] fp16; slot_mapping: [T] int64;
    k_cache, v_cache: [NB, Hk, bs, d] fp16.  Returns (k_cache', v_cache').
    Raises OracleError when a slot lies beyond the pool.
    """
    kc, vc = _u16(k_cache).copy(), _u16(v_cache).copy()
    append_inplace(k_new, v_new, slot_mapping, kc, vc, block_size, lib=lib)
    return kc.view(np.float16), vc.view(np.float16)


def append_inplace(k_new, v_new, slot_mapping, k_cache, v_cache, block_size, lib=None):
    """The same append, written into k_cache / v_cache themselves (contiguous
    fp16 or uint16 arrays, modified in place)."""
    lib = lib or load()
    k_new, v_new = _u16(k_new), _u16(v_new)
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.flags.c_contiguous
                and c.dtype in (np.float16, np.uint16)):
            raise TypeError("caches must be contiguous fp16/uint16 arrays")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hk, d = k_new.shape
    NB, Hk2, bs, d2 = k_cache.shape
    if (Hk2, d2, bs) != (Hk, d, block_size) or v_new.shape != k_new.shape or \
            v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    rc = lib.pkvo_append(_ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(k_cache), _ptr(v_cache), T,
                         Hk, d, bs, NB)
    if rc != 0:
        raise OracleError("slot beyond the pool")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, n_q_heads, n_kv_heads,
           head_dim, block_size, mask=None, num_threads=0, lib=None):
    """Paged decode attention.  Returns (out f64 [B,H,d], lse f64 [B,H], out fp16 [B,H,d]).

    q: [B, H, d] fp16; caches [NB, Hk, bs, d] fp16; block_tables [B, MB] int32;
    context_lens [B] int32; mask: optional bool [B, H] selecting the pairs to
    compute (the others stay NaN).
    """
    lib = lib or load()
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, d = q.shape
    NB = kc.shape[0]
    if (H, d) != (n_q_heads, head_dim) or kc.shape != (NB, n_kv_heads, block_size, head_dim):
        raise ValueError("shape mismatch")
    if vc.shape != kc.shape or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("shape mismatch")
    MB = bt.shape[1]
    out = np.full((B, H, d), np.nan)
    lse = np.full((B, H), np.nan)
    out16 = np.zeros((B, H, d), dtype=np.uint16)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8).reshape(B * H)
    rc = lib.pkvo_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), B, MB, NB,
                         float(scale), n_q_heads, n_kv_heads, head_dim, block_size, _ptr(m),
                         _ptr(out), _ptr(lse), _ptr(out16), int(num_threads))
    if rc != 0:
        raise OracleError("invalid decode input")
    return out, lse, out16.view(np.float16)


def partial(q, k_cache, v_cache, block_tables, scale, n_q_heads, n_kv_heads, head_dim,
            block_size, b, h, t_begin, t_end, lib=None):
    """(m, l, acc) of one (b, h) over tokens [t_begin, t_end) (acc not normalised)."""
    lib = lib or load()
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(head_dim)
    rc = lib.pkvo_decode_partial(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                 kc.shape[0], float(scale), n_q_heads, n_kv_heads, head_dim,
                                 block_size, int(b), int(h), int(t_begin), int(t_end), _ptr(m),
                                 _ptr(l), _ptr(acc))
    if rc != 0:
        raise OracleError("invalid partial input")
    return float(m[0]), float(l[0]), acc


def lse_merge(m, l, acc, lib=None):
    """Merge partials: m [n], l [n], acc [n, d] -> (out [d], lse)."""
    lib = lib or load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    n, d = acc.shape
    out = np.zeros(d)
    lse = np.zeros(1)
    lib.pkvo_lse_merge(n, _ptr(m), _ptr(l), _ptr(acc), d, _ptr(out), _ptr(lse))
    return out, float(lse[0])


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# ---------------------------------------------------------------------------

def e4m3_to_f64(code: int, lib=None) -> float:
    """Value of one E4M3 code (NaN for 0x7f / 0xff)."""
    return (lib or load()).pkvo_e4m3_to_f64(int(code))


def e4m3_table(lib=None):
    """Values of all 256 codes, float64 [256]."""
    lib = lib or load()
    return np.array([lib.pkvo_e4m3_to_f64(i) for i in range(256)])


def f32_to_e4m3(y, lib=None):
    """E4M3 codes (uint8) of fp32 values: nearest, ties to even, saturating."""
    lib = lib or load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.zeros(y.shape, dtype=np.uint8)
    lib.pkvo_f32_to_e4m3_array(_ptr(y), y.size, _ptr(out))
    return out


def quantize_e4m3(x16, scale, lib=None):
    """Codes of fp16 values under a scale: E4M3(fp32(x) / fp32(scale))."""
    lib = lib or load()
    x = _u16(x16)
    out = np.zeros(x.shape, dtype=np.uint8)
    lib.pkvo_quantize_e4m3_array(_ptr(x), x.size, float(np.float32(scale)), _ptr(out))
    return out


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8 codes, got {a.dtype}")
    return a


def append_f8(k_new, v_new, slot_mapping, k_cache8, v_cache8, block_size, k_scale, v_scale,
              lib=None):
    """Slot-mapped append into copies of FP8 caches ([NB, Hk, bs, d] uint8 codes)."""
    lib = lib or load()
    k_new, v_new = _u16(k_new), _u16(v_new)
    kc, vc = _u8(k_cache8).copy(), _u8(v_cache8).copy()
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hk, d = k_new.shape
    NB, Hk2, bs, d2 = kc.shape
    if (Hk2, d2, bs) != (Hk, d, block_size) or v_new.shape != k_new.shape or vc.shape != kc.shape:
        raise ValueError("shape mismatch")
    rc = lib.pkvo_append_f8(_ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(kc), _ptr(vc), T, Hk,
                            d, bs, NB, float(np.float32(k_scale)), float(np.float32(v_scale)))
    if rc != 0:
        raise OracleError("slot beyond the pool")
    return kc, vc


def decode_f8(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, context_lens, scale,
              n_q_heads, n_kv_heads, head_dim, block_size, mask=None, num_threads=0, lib=None):
    """Paged decode attention over FP8 caches.  Returns (out f64 [B,H,d], lse f64 [B,H])."""
    lib = lib or load()
    q = _u16(q)
    kc, vc = _u8(k_cache8), _u8(v_cache8)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, d = q.shape
    NB = kc.shape[0]
    if (H, d) != (n_q_heads, head_dim) or kc.shape != (NB, n_kv_heads, block_size, head_dim):
        raise ValueError("shape mismatch")
    if vc.shape != kc.shape or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("shape mismatch")
    out = np.full((B, H, d), np.nan)
    lse = np.full((B, H), np.nan)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8).reshape(B * H)
    rc = lib.pkvo_decode_f8(_ptr(q), _ptr(kc), _ptr(vc), float(np.float32(k_scale)),
                            float(np.float32(v_scale)), _ptr(bt), _ptr(cl), B, bt.shape[1], NB,
                            float(scale), n_q_heads, n_kv_heads, head_dim, block_size, _ptr(m),
                            _ptr(out), _ptr(lse), int(num_threads))
    if rc != 0:
        raise OracleError("invalid decode input")
    return out, lse


# ---------------------------------------------------------------------------
# multi-token (causal) paged attention
# ---------------------------------------------------------------------------

def decode_multi(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                 n_q_heads, n_kv_heads, head_dim, block_size, num_threads=0, lib=None):
    """Causal attention of each sequence's last n_b tokens over its paged K/V.

    q: [total_q, H, d] fp16, query rows [query_start[b], query_start[b+1]) of
    sequence b at positions L_b - n_b + i.  Returns (out f64 [total_q, H, d],
    lse f64 [total_q, H]).
    """
    lib = lib or load()
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    B = cl.shape[0]
    TQ, H, d = q.shape
    NB = kc.shape[0]
    if (H, d) != (n_q_heads, head_dim) or kc.shape != (NB, n_kv_heads, block_size, head_dim):
        raise ValueError("shape mismatch")
    if vc.shape != kc.shape or bt.shape[0] != B or qs.shape != (B + 1,) or qs[-1] != TQ:
        raise ValueError("shape mismatch")
    out = np.full((TQ, H, d), np.nan)
    lse = np.full((TQ, H), np.nan)
    rc = lib.pkvo_decode_multi(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), _ptr(qs), B,
                               bt.shape[1], NB, float(scale), n_q_heads, n_kv_heads, head_dim,
                               block_size, _ptr(out), _ptr(lse), int(num_threads))
    if rc != 0:
        raise OracleError("invalid multi-token input")
    return out, lse
