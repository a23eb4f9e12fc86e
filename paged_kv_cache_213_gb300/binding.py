"""ctypes binding of ``libpagedkv.so`` (the C ABI in ``include/pagedkv.h``).

Argument marshalling only: shapes, dtypes, device and contiguity checks,
data pointers, the current torch stream, and torch allocation of outputs and
workspace.  Every step of the computation runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing, or a tensor
is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_WORKSPACE = -3
PKV_ERR_CUDA = -4
PKV_ERR_INDEX = -5

PKV_ERRBIT_BLOCK_ID = 0x1
PKV_ERRBIT_SLOT = 0x2
PKV_ERRBIT_CONTEXT = 0x4
PKV_ERRBIT_TIMEOUT = 0x8
PKV_ERRBIT_WORKSPACE = 0x10
PKV_ERRBIT_APPEND = 0x20
# bytes at the start of a workspace that hold arrival counters and must be
# zero when a call starts
PKV_WORKSPACE_COUNTER_BYTES = 65536

_lock = threading.Lock()
_lib = None


class PagedKVError(RuntimeError):
    """A library call returned a negative status."""

    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def library():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it first "
                "(python -m paged_kv_cache_213_gb300.build, or __graft_entry__.build())")
        lib = ctypes.CDLL(_LIB_PATH)
        c = ctypes
        p = c.c_void_p
        lib.paged_kv_append.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int,
                                        c.c_int64, p, p]
        lib.paged_kv_append.restype = c.c_int
        lib.paged_decode_plan.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                          c.c_int, c.c_int, c.POINTER(c.c_int),
                                          c.POINTER(c.c_size_t)]
        lib.paged_decode_plan.restype = c.c_int
        lib.paged_decode_attention.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64,
                                               c.c_float, c.c_int, c.c_int, c.c_int, c.c_int,
                                               c.c_int, c.c_int, p, c.c_size_t, p, p, p]
        lib.paged_decode_attention.restype = c.c_int
        lib.paged_decode_attention_ex.argtypes = lib.paged_decode_attention.argtypes + [c.c_uint32]
        lib.paged_decode_attention_ex.restype = c.c_int
        lib.paged_decode_workspace_clear.argtypes = [p, c.c_size_t, p]
        lib.paged_decode_workspace_clear.restype = c.c_int
        lib.paged_kv_get_error.argtypes = [p, p, c.POINTER(c.c_int32)]
        lib.paged_kv_get_error.restype = c.c_int
        lib.paged_kv_status_string.argtypes = [c.c_int]
        lib.paged_kv_status_string.restype = c.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return library().paged_kv_status_string(int(status)).decode()


def _check(func: str, status: int):
    if status != PKV_OK:
        raise PagedKVError(func, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _need_out(out, dev):
    """out: fp16 on the call's device, or a pinned host tensor, which the
    kernels write directly (plain stores into mapped host memory)."""
    if isinstance(out, torch.Tensor) and not out.is_cuda and out.is_pinned():
        if out.dtype != torch.float16:
            raise TypeError(f"out must be {torch.float16}, got {out.dtype}")
        if not out.is_contiguous():
            raise ValueError("out must be contiguous")
        return
    _need(out, "out", torch.float16, dev)


def paged_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, err_word=None):
    """Write k_new/v_new [T, Hk, d] (fp16) into slots slot_mapping [T] (int64)
    of k_cache/v_cache [NB, Hk, bs, d] (fp16), in place, on the current stream."""
    dev = k_cache.device
    _need(k_new, "k_new", torch.float16, dev)
    _need(v_new, "v_new", torch.float16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    _need(k_cache, "k_cache", torch.float16, dev)
    _need(v_cache, "v_cache", torch.float16, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must both be [num_blocks, n_kv_heads, block_size, head_dim]")
    NB, Hk, bs, d = k_cache.shape
    if k_new.dim() != 3 or k_new.shape[1:] != (Hk, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens, n_kv_heads, head_dim]")
    T = k_new.shape[0]
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    with torch.cuda.device(dev):
        rc = library().paged_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                       _ptr(k_cache), _ptr(v_cache), T, Hk, d, bs, NB,
                                       _ptr(err_word), _stream_handle(dev))
    _check("paged_kv_append", rc)


def decode_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                max_context_len=0, partition_tokens=0):
    """(partition_tokens, workspace_bytes) the library will use."""
    P = ctypes.c_int(0)
    W = ctypes.c_size_t(0)
    rc = library().paged_decode_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                     max_blocks_per_seq, max_context_len, partition_tokens,
                                     ctypes.byref(P), ctypes.byref(W))
    _check("paged_decode_plan", rc)
    return P.value, W.value


PKV_TABLES_READY = 0x1
PKV_APPEND_NEWEST = 0x2  # paged_decode_step: token b is sequence b's newest (one launch)


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, n_q_heads,
                           n_kv_heads, head_dim, block_size, max_context_len=None,
                           partition_tokens=0, out=None, workspace=None, lse=None,
                           err_word=None, flags=0):
    """softmax(q K^T * scale) V over each sequence's paged K/V -> out [B, H, d] fp16.

    q [B, H, d] fp16; k_cache/v_cache [NB, Hk, bs, d] fp16; block_tables
    [B, MB] int32; context_lens [B] int32.  max_context_len: an upper bound on
    context_lens (None -> MB * bs; pass the host-side value to keep the launch
    free of a device sync).  lse: optional fp32 [B, H] output tensor.
    flags: 0 (paged_decode_attention) or PKV_TABLES_READY
    (paged_decode_attention_ex: the kernel launched just before on the
    current stream writes neither context_lens nor block_tables).
    """
    dev = q.device
    _need(q, "q", torch.float16, dev)
    _need(k_cache, "k_cache", torch.float16, dev)
    _need(v_cache, "v_cache", torch.float16, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    B = q.shape[0]
    if q.dim() != 3 or q.shape[1:] != (n_q_heads, head_dim):
        raise ValueError("q must be [num_seqs, n_q_heads, head_dim]")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or \
            k_cache.shape[1:] != (n_kv_heads, block_size, head_dim):
        raise ValueError("caches must be [num_blocks, n_kv_heads, block_size, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, MB], context_lens [B]")
    MB = block_tables.shape[1]
    mcl = 0 if max_context_len is None else int(max_context_len)
    P, ws_bytes = decode_plan(B, n_q_heads, n_kv_heads, head_dim, block_size, MB, mcl,
                              partition_tokens)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_out(out, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
        if lse.shape != (B, n_q_heads):
            raise ValueError("lse must be [B, H]")
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    if ws_bytes > 0:
        if workspace is None:
            # zero-filled: the balanced split keeps arrival counters in it
            workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        else:
            _need(workspace, "workspace", torch.uint8, dev)
    args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), B, MB, k_cache.shape[0], float(scale), n_q_heads, n_kv_heads,
            head_dim, block_size, mcl, P, _ptr(workspace) if ws_bytes > 0 else None,
            workspace.numel() if (ws_bytes > 0) else 0, _ptr(lse), _ptr(err_word))
    with torch.cuda.device(dev):
        if flags:
            rc = library().paged_decode_attention_ex(*args, _stream_handle(dev), int(flags))
        else:
            rc = library().paged_decode_attention(*args, _stream_handle(dev))
    _check("paged_decode_attention_ex" if flags else "paged_decode_attention", rc)
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale,
                                   n_q_heads, n_kv_heads, head_dim, block_size,
                                   max_context_len=None, partition_tokens=0, out=None, lse=None,
                                   err_word=None):
    """Like paged_decode_attention, but the split-K scratch is the library's
    static device array, for callers that cannot allocate device memory.
    ``out`` (and ``lse``) should be passed in by such callers; calls whose
    kernels overlap on the GPU race on the shared scratch."""
    lib = library()
    fn = lib.paged_decode_attention_noalloc
    if fn.restype is not ctypes.c_int:
        c = ctypes
        p = c.c_void_p
        fn.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float, c.c_int,
                       c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p, p, p]
        fn.restype = c.c_int
    dev = q.device
    for t, name, dt in ((q, "q", torch.float16), (k_cache, "k_cache", torch.float16),
                        (v_cache, "v_cache", torch.float16),
                        (block_tables, "block_tables", torch.int32),
                        (context_lens, "context_lens", torch.int32)):
        _need(t, name, dt, dev)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    B, MB = block_tables.shape
    mcl = 0 if max_context_len is None else int(max_context_len)
    with torch.cuda.device(dev):
        rc = fn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                _ptr(context_lens), B, MB, k_cache.shape[0], float(scale), n_q_heads, n_kv_heads,
                head_dim, block_size, mcl, int(partition_tokens), _ptr(lse), _ptr(err_word),
                _stream_handle(dev))
    _check("paged_decode_attention_noalloc", rc)
    return out


def paged_copy_in(dst: torch.Tensor, src: torch.Tensor):
    """dst (device) <- src (device or pinned host) by a library kernel, on the
    current stream: both contiguous uint8 of the same size, a multiple of 16."""
    _need(dst, "dst", torch.uint8)
    if not (isinstance(src, torch.Tensor) and (src.is_cuda or src.is_pinned())):
        raise ValueError("src must be a CUDA tensor or pinned host memory")
    if src.dtype != torch.uint8 or not src.is_contiguous() or src.numel() != dst.numel():
        raise ValueError("src must be contiguous uint8 of dst's size")
    lib = library()
    fn = lib.paged_copy_in
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    with torch.cuda.device(dst.device):
        _check("paged_copy_in", fn(_ptr(dst), _ptr(src), dst.numel(),
                                   _stream_handle(dst.device)))


def paged_decode_workspace_clear(workspace: torch.Tensor):
    """Zero a workspace's arrival counters on the current stream (needed after a
    call flagged PKV_ERRBIT_TIMEOUT or PKV_ERRBIT_WORKSPACE)."""
    _need(workspace, "workspace", torch.uint8)
    with torch.cuda.device(workspace.device):
        _check("paged_decode_workspace_clear",
               library().paged_decode_workspace_clear(
                   _ptr(workspace) if workspace.numel() else None, workspace.numel(),
                   _stream_handle(workspace.device)))


def get_error(err_word: torch.Tensor) -> int:
    """Wait for the current stream and return the device error word's bits."""
    _need(err_word, "err_word", torch.int32)
    bits = ctypes.c_int32(0)
    with torch.cuda.device(err_word.device):
        rc = library().paged_kv_get_error(_ptr(err_word), _stream_handle(err_word.device),
                                          ctypes.byref(bits))
    if rc not in (PKV_OK, PKV_ERR_INDEX):
        _check("paged_kv_get_error", rc)
    return int(bits.value)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def _prefix_shared_plan(name, num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                        max_blocks_per_seq, max_context_len, num_groups, max_group_size,
                        max_prefix_len):
    lib = library()
    fn = getattr(lib, name)
    c = ctypes
    fn.argtypes = [c.c_int] * 10 + [c.POINTER(c.c_size_t)]
    fn.restype = c.c_int
    W = c.c_size_t(0)
    _check(name, fn(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                    max_context_len, num_groups, max_group_size, max_prefix_len, c.byref(W)))
    return W.value


def prefix_shared_plan(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                       max_context_len, num_groups, max_group_size, max_prefix_len):
    """Workspace bytes of paged_decode_attention_prefix_shared."""
    return _prefix_shared_plan("paged_decode_prefix_shared_plan", num_seqs, n_q_heads,
                               n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                               max_context_len, num_groups, max_group_size, max_prefix_len)


def prefix_shared_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, max_context_len, num_groups, max_group_size,
                           max_prefix_len):
    """Workspace bytes of paged_decode_attention_prefix_shared_fp8."""
    return _prefix_shared_plan("paged_decode_prefix_shared_plan_fp8", num_seqs, n_q_heads,
                               n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                               max_context_len, num_groups, max_group_size, max_prefix_len)


def _prefix_shared_call(scales, q, k_cache, v_cache, block_tables, context_lens, scale,
                        n_q_heads, n_kv_heads, head_dim, block_size, group_offsets,
                        group_prefix_lens, max_group_size, max_prefix_len, max_context_len, out,
                        workspace, lse, err_word, flags=0):
    """scales: None (fp16 caches) or (k_scale, v_scale) of E4M3 caches;
    flags: launch flags (the _ex entry points)."""
    fp8 = scales is not None
    name = "paged_decode_attention_prefix_shared" + ("_fp8" if fp8 else "") + \
        ("_ex" if flags else "")
    lib = library()
    fn = getattr(lib, name)
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float] + \
        ([c.c_float, c.c_float] if fp8 else []) + \
        [c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p, p, c.c_int, c.c_int, c.c_int, p,
         c.c_size_t, p, p, p] + ([c.c_uint32] if flags else [])
    fn.restype = c.c_int
    dev = q.device
    kv_dtype = torch.uint8 if fp8 else torch.float16
    for t, nm, dt in ((q, "q", torch.float16), (k_cache, "k_cache", kv_dtype),
                      (v_cache, "v_cache", kv_dtype),
                      (block_tables, "block_tables", torch.int32),
                      (context_lens, "context_lens", torch.int32),
                      (group_offsets, "group_offsets", torch.int32),
                      (group_prefix_lens, "group_prefix_lens", torch.int32)):
        _need(t, nm, dt, dev)
    B, MB = block_tables.shape
    G = group_prefix_lens.numel()
    if group_offsets.numel() != G + 1:
        raise ValueError("group_offsets must have num_groups + 1 entries")
    mcl = 0 if max_context_len is None else int(max_context_len)
    ws = _prefix_shared_plan("paged_decode_prefix_shared_plan" + ("_fp8" if fp8 else ""), B,
                             n_q_heads, n_kv_heads, head_dim, block_size, MB, mcl, G,
                             max_group_size, max_prefix_len)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.float16, dev)
    if workspace is None:
        # zero-filled: the balanced split keeps arrival counters in it
        workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    extra = [float(scales[0]), float(scales[1])] if fp8 else []
    with torch.cuda.device(dev):
        rc = fn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                _ptr(context_lens), B, MB, k_cache.shape[0], float(scale), *extra, n_q_heads,
                n_kv_heads, head_dim, block_size, mcl, _ptr(group_offsets),
                _ptr(group_prefix_lens), G, int(max_group_size), int(max_prefix_len),
                _ptr(workspace), workspace.numel(), _ptr(lse), _ptr(err_word),
                _stream_handle(dev), *([int(flags)] if flags else []))
    _check(name, rc)
    return out


def paged_decode_attention_prefix_shared(q, k_cache, v_cache, block_tables, context_lens, scale,
                                         n_q_heads, n_kv_heads, head_dim, block_size,
                                         group_offsets, group_prefix_lens, max_group_size,
                                         max_prefix_len, max_context_len=None, out=None,
                                         workspace=None, lse=None, err_word=None, flags=0):
    """Decode attention that reads each group's shared prefix blocks once per
    chunk of members.  group_offsets [G+1] and group_prefix_lens [G] are int32
    CUDA tensors (consecutive ranges of sequences, shared prefix tokens).
    flags: 0, or PKV_TABLES_READY (paged_decode_attention_prefix_shared_ex)."""
    return _prefix_shared_call(None, q, k_cache, v_cache, block_tables, context_lens, scale,
                               n_q_heads, n_kv_heads, head_dim, block_size, group_offsets,
                               group_prefix_lens, max_group_size, max_prefix_len,
                               max_context_len, out, workspace, lse, err_word, flags)


def paged_decode_attention_prefix_shared_fp8(q, k_cache, v_cache, block_tables, context_lens,
                                             scale, k_scale, v_scale, n_q_heads, n_kv_heads,
                                             head_dim, block_size, group_offsets,
                                             group_prefix_lens, max_group_size, max_prefix_len,
                                             max_context_len=None, out=None, workspace=None,
                                             lse=None, err_word=None, flags=0):
    """The prefix-aware call over E4M3 caches (uint8 codes; values code *
    k_scale and code * v_scale).  flags: 0, or PKV_TABLES_READY."""
    return _prefix_shared_call((k_scale, v_scale), q, k_cache, v_cache, block_tables,
                               context_lens, scale, n_q_heads, n_kv_heads, head_dim, block_size,
                               group_offsets, group_prefix_lens, max_group_size, max_prefix_len,
                               max_context_len, out, workspace, lse, err_word, flags)


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV caches: uint8 tensors of codes, one scale per cache tensor
# ---------------------------------------------------------------------------

def paged_kv_append_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                        err_word=None):
    """Quantize k_new/v_new [T, Hk, d] (fp16) to E4M3 codes (x / scale, nearest-even,
    saturating) into slots of k_cache/v_cache [NB, Hk, bs, d] (uint8), in place."""
    lib = library()
    fn = lib.paged_kv_append_fp8
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64, c.c_float,
                   c.c_float, p, p]
    fn.restype = c.c_int
    dev = k_cache.device
    _need(k_new, "k_new", torch.float16, dev)
    _need(v_new, "v_new", torch.float16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    _need(k_cache, "k_cache", torch.uint8, dev)
    _need(v_cache, "v_cache", torch.uint8, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must both be [num_blocks, n_kv_heads, block_size, head_dim]")
    NB, Hk, bs, d = k_cache.shape
    if k_new.dim() != 3 or k_new.shape[1:] != (Hk, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens, n_kv_heads, head_dim]")
    T = k_new.shape[0]
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    with torch.cuda.device(dev):
        rc = fn(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), T,
                Hk, d, bs, NB, float(k_scale), float(v_scale), _ptr(err_word),
                _stream_handle(dev))
    _check("paged_kv_append_fp8", rc)


def decode_plan_fp8(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                    max_context_len=0):
    """Workspace bytes of paged_decode_attention_fp8."""
    lib = library()
    fn = lib.paged_decode_plan_fp8
    c = ctypes
    fn.argtypes = [c.c_int] * 7 + [c.POINTER(c.c_size_t)]
    fn.restype = c.c_int
    W = c.c_size_t(0)
    _check("paged_decode_plan_fp8",
           fn(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
              max_context_len, c.byref(W)))
    return W.value


def paged_decode_attention_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale,
                               v_scale, n_q_heads, n_kv_heads, head_dim, block_size,
                               max_context_len=None, out=None, workspace=None, lse=None,
                               err_word=None, flags=0):
    """Decode attention over E4M3 caches [NB, Hk, bs, d] (uint8): keys and values are
    code * k_scale and code * v_scale.  Returns out [B, H, d] fp16.  flags: 0, or
    PKV_TABLES_READY (paged_decode_attention_fp8_ex)."""
    lib = library()
    name = "paged_decode_attention_fp8" + ("_ex" if flags else "")
    fn = getattr(lib, name)
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float, c.c_float,
                   c.c_float, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p, c.c_size_t, p, p,
                   p] + ([c.c_uint32] if flags else [])
    fn.restype = c.c_int
    dev = q.device
    _need(q, "q", torch.float16, dev)
    _need(k_cache, "k_cache", torch.uint8, dev)
    _need(v_cache, "v_cache", torch.uint8, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    B = q.shape[0]
    if q.dim() != 3 or q.shape[1:] != (n_q_heads, head_dim):
        raise ValueError("q must be [num_seqs, n_q_heads, head_dim]")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or \
            k_cache.shape[1:] != (n_kv_heads, block_size, head_dim):
        raise ValueError("caches must be [num_blocks, n_kv_heads, block_size, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, MB], context_lens [B]")
    MB = block_tables.shape[1]
    mcl = 0 if max_context_len is None else int(max_context_len)
    ws = decode_plan_fp8(B, n_q_heads, n_kv_heads, head_dim, block_size, MB, mcl)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.float16, dev)
    if workspace is None:
        # zero-filled: the balanced split keeps arrival counters in it
        workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        rc = fn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                _ptr(context_lens), B, MB, k_cache.shape[0], float(scale), float(k_scale),
                float(v_scale), n_q_heads, n_kv_heads, head_dim, block_size, mcl,
                _ptr(workspace), workspace.numel(), _ptr(lse), _ptr(err_word),
                _stream_handle(dev), *([int(flags)] if flags else []))
    _check(name, rc)
    return out


def paged_decode_step_fp8(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                          context_lens, scale, k_scale, v_scale, n_q_heads, n_kv_heads,
                          head_dim, block_size, max_context_len=None, out=None, workspace=None,
                          lse=None, err_word=None, flags=0):
    """One decode step over E4M3 caches: paged_kv_append_fp8 then
    paged_decode_attention_fp8 in one call.  flags (paged_decode_step_fp8_ex):
    PKV_APPEND_NEWEST (token b is sequence b's newest: the attention kernel
    quantizes and appends it, one launch) and PKV_TABLES_READY.  Returns out."""
    lib = library()
    fn = lib.paged_decode_step_fp8_ex
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, c.c_int, p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float,
                   c.c_float, c.c_float, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p,
                   c.c_size_t, p, p, p, c.c_uint32]
    fn.restype = c.c_int
    dev = q.device
    for t, name, dt in ((k_new, "k_new", torch.float16), (v_new, "v_new", torch.float16),
                        (slot_mapping, "slot_mapping", torch.int64), (q, "q", torch.float16),
                        (k_cache, "k_cache", torch.uint8), (v_cache, "v_cache", torch.uint8),
                        (block_tables, "block_tables", torch.int32),
                        (context_lens, "context_lens", torch.int32)):
        _need(t, name, dt, dev)
    B, MB = block_tables.shape
    T = k_new.shape[0]
    if slot_mapping.shape != (T,) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new [T, Hk, d], slot_mapping [T]")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or \
            k_cache.shape[1:] != (n_kv_heads, block_size, head_dim):
        raise ValueError("caches must be [num_blocks, n_kv_heads, block_size, head_dim]")
    mcl = 0 if max_context_len is None else int(max_context_len)
    ws = decode_plan_fp8(B, n_q_heads, n_kv_heads, head_dim, block_size, MB, mcl)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.float16, dev)
    if workspace is None:
        # zero-filled: the balanced split keeps arrival counters in it
        workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        rc = fn(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(out), _ptr(q),
                _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, MB,
                k_cache.shape[0], float(scale), float(k_scale), float(v_scale), n_q_heads,
                n_kv_heads, head_dim, block_size, mcl, _ptr(workspace), workspace.numel(),
                _ptr(lse), _ptr(err_word), _stream_handle(dev), int(flags))
    _check("paged_decode_step_fp8_ex", rc)
    return out


# ---------------------------------------------------------------------------
# multi-token (causal) attention: speculative verify, chunked prefill
# ---------------------------------------------------------------------------

def step_launches(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                  max_context_len=0, partition_tokens=0, num_tokens=None, flags=0):
    """Kernels that paged_decode_step launches for these sizes and flags."""
    lib = library()
    fn = lib.paged_decode_step_launches
    c = ctypes
    fn.argtypes = [c.c_int] * 9 + [c.c_uint32, c.POINTER(c.c_int)]
    fn.restype = c.c_int
    n = ctypes.c_int(-1)
    _check("paged_decode_step_launches",
           fn(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq,
              int(max_context_len or 0), partition_tokens,
              num_seqs if num_tokens is None else num_tokens, int(flags), ctypes.byref(n)))
    return n.value


def multi_plan(num_seqs, total_q, max_q_len, n_q_heads, n_kv_heads, head_dim, block_size,
               max_blocks_per_seq, max_context_len=0, partition_tokens=0):
    """(partition_tokens, workspace_bytes) of paged_decode_attention_multi."""
    lib = library()
    fn = lib.paged_decode_multi_plan
    c = ctypes
    fn.argtypes = [c.c_int] * 10 + [c.POINTER(c.c_int), c.POINTER(c.c_size_t)]
    fn.restype = c.c_int
    P = c.c_int(0)
    W = c.c_size_t(0)
    _check("paged_decode_multi_plan",
           fn(num_seqs, total_q, max_q_len, n_q_heads, n_kv_heads, head_dim, block_size,
              max_blocks_per_seq, max_context_len, partition_tokens, c.byref(P), c.byref(W)))
    return P.value, W.value


def paged_decode_attention_multi(q, k_cache, v_cache, block_tables, context_lens, query_start,
                                 scale, n_q_heads, n_kv_heads, head_dim, block_size, max_q_len,
                                 max_context_len=None, partition_tokens=0, out=None,
                                 workspace=None, lse=None, err_word=None, flags=0):
    """Causal attention of each sequence's last n_b tokens over its paged K/V.

    q [total_q, H, d] fp16 (sequence b owns rows [query_start[b], query_start[b+1]));
    query_start [B + 1] int32; context_lens include the new tokens.  Returns
    out [total_q, H, d] fp16.  flags: 0, or PKV_TABLES_READY
    (paged_decode_attention_multi_ex; the promise covers query_start)."""
    lib = library()
    name = "paged_decode_attention_multi" + ("_ex" if flags else "")
    fn = getattr(lib, name)
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64, c.c_float,
                   c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p, c.c_size_t, p, p,
                   p] + ([c.c_uint32] if flags else [])
    fn.restype = c.c_int
    dev = q.device
    for t, name, dt in ((q, "q", torch.float16), (k_cache, "k_cache", torch.float16),
                        (v_cache, "v_cache", torch.float16),
                        (block_tables, "block_tables", torch.int32),
                        (context_lens, "context_lens", torch.int32),
                        (query_start, "query_start", torch.int32)):
        _need(t, name, dt, dev)
    B, MB = block_tables.shape
    TQ = q.shape[0]
    if q.dim() != 3 or q.shape[1:] != (n_q_heads, head_dim):
        raise ValueError("q must be [total_q, n_q_heads, head_dim]")
    if query_start.shape != (B + 1,) or context_lens.shape != (B,):
        raise ValueError("query_start must be [B + 1], context_lens [B]")
    mcl = 0 if max_context_len is None else int(max_context_len)
    P, ws = multi_plan(B, TQ, int(max_q_len), n_q_heads, n_kv_heads, head_dim, block_size, MB,
                       mcl, partition_tokens)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.float16, dev)
    if ws > 0:
        if workspace is None:
            # zero-filled: the balanced split keeps arrival counters in it
            workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        rc = fn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                _ptr(context_lens), _ptr(query_start), B, TQ, int(max_q_len), MB,
                k_cache.shape[0], float(scale), n_q_heads, n_kv_heads, head_dim, block_size, mcl,
                P, _ptr(workspace) if ws > 0 else None, workspace.numel() if ws > 0 else 0,
                _ptr(lse), _ptr(err_word), _stream_handle(dev), *([int(flags)] if flags else []))
    _check(name, rc)
    return out


def paged_decode_step(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                      context_lens, scale, n_q_heads, n_kv_heads, head_dim, block_size,
                      max_context_len=None, partition_tokens=0, out=None, workspace=None,
                      lse=None, err_word=None, flags=0):
    """paged_kv_append then paged_decode_attention in one call: the attention's
    prologue overlaps the append.  flags (paged_decode_step_ex):
    PKV_APPEND_NEWEST (token b is sequence b's newest: the attention kernel
    appends it, one launch) and PKV_TABLES_READY.  Returns out [B, H, d] fp16."""
    lib = library()
    fn = lib.paged_decode_step_ex
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, c.c_int, p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float,
                   c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p, c.c_size_t, p, p, p,
                   c.c_uint32]
    fn.restype = c.c_int
    dev = q.device
    for t, name, dt in ((k_new, "k_new", torch.float16), (v_new, "v_new", torch.float16),
                        (slot_mapping, "slot_mapping", torch.int64), (q, "q", torch.float16),
                        (k_cache, "k_cache", torch.float16), (v_cache, "v_cache", torch.float16),
                        (block_tables, "block_tables", torch.int32),
                        (context_lens, "context_lens", torch.int32)):
        _need(t, name, dt, dev)
    B, MB = block_tables.shape
    T = k_new.shape[0]
    if slot_mapping.shape != (T,) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new [T, Hk, d], slot_mapping [T]")
    mcl = 0 if max_context_len is None else int(max_context_len)
    P, ws = decode_plan(B, n_q_heads, n_kv_heads, head_dim, block_size, MB, mcl, partition_tokens)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_out(out, dev)
    if ws > 0:
        if workspace is None:
            # zero-filled: the balanced split keeps arrival counters in it
            workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        rc = fn(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(out), _ptr(q),
                _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), B, MB,
                k_cache.shape[0], float(scale), n_q_heads, n_kv_heads, head_dim, block_size, mcl,
                P, _ptr(workspace) if ws > 0 else None, workspace.numel() if ws > 0 else 0,
                _ptr(lse), _ptr(err_word), _stream_handle(dev), int(flags))
    _check("paged_decode_step_ex", rc)
    return out
