"""The allocation-free entry point gives the same results as the regular one.

paged_decode_attention_noalloc is for callers that cannot allocate device
memory -- an operator inside a host framework's plugin interface that gets its
tensors but no allocator, or a foreign-language binding without a CUDA
allocator -- and so cannot pass the split-K workspace.  It keeps that scratch
in a static array inside the library.  Here it is called through the C ABI
several times in a row: the balanced split (the default, whose arrival
counters live at the start of the array and must be zero when a call starts)
before and after fixed-partition calls on the same array, and on problems of
different shapes.  Each result is compared with paged_decode_attention given
a caller-allocated workspace and with the CPU oracle.  This file is collected
last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_213_gb300 as pkv
from gpu_util import MAX_ABS, REL_L2, compare, oracle_step, to_dev
from paged_kv_cache_213_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _c_noalloc():
    fn = pkv.library().paged_decode_attention_noalloc
    c = ctypes
    p = c.c_void_p
    fn.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float, c.c_int, c.c_int,
                   c.c_int, c.c_int, c.c_int, c.c_int, p, p, p]
    fn.restype = c.c_int
    return fn


def _prepare(batch):
    dev = to_dev(batch)
    if batch.has_append:
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"])
    return dev


def _regular(batch, dev, P):
    return pkv.paged_decode_attention(
        dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
        batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
        max_context_len=batch.max_context_len, partition_tokens=P)


def _noalloc(fn, batch, dev, P):
    """One call through the C ABI into NaN-filled out / lse (every output the
    call owes must be written)."""
    out = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = fn(p(out), p(dev["q"]), p(dev["k_cache"]), p(dev["v_cache"]), p(dev["block_tables"]),
            p(dev["context_lens"]), batch.num_seqs, batch.max_blocks_per_seq, batch.num_blocks,
            batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
            batch.max_context_len, P, p(lse), p(err), stream)
    assert rc == 0, pkv.status_string(rc)
    return out, lse, err


def test_noalloc_matches_regular_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _c_noalloc()
    big = wl.workload(2, poison=True)
    small = wl.workload(1, poison=True)
    # balanced, fixed partitions on the same array, balanced again, then
    # another shape both ways: consecutive calls share the array
    cases = [(big, 0), (big, 256), (big, 0), (small, 16), (small, 0), (big, 0)]
    for batch, P in cases:
        _, need = pkv.decode_plan(batch.num_seqs, batch.n_q_heads, batch.n_kv_heads,
                                  batch.head_dim, batch.block_size, batch.max_blocks_per_seq,
                                  batch.max_context_len, P)
        assert 0 < need <= pkv.binding.NOALLOC_SCRATCH_BYTES
    devs = {id(big): _prepare(big), id(small): _prepare(small)}
    oracles = {id(b): oracle_step(b)["out"] for b in (big, small)}
    refs = [_regular(b, devs[id(b)], P) for b, P in cases]
    got = [_noalloc(fn, b, devs[id(b)], P) for b, P in cases]
    torch.cuda.synchronize()
    for (b, P), ref, (out, lse, err) in zip(cases, refs, got):
        assert pkv.get_error(err) == 0, (b.name, P)
        out_np = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(out_np)), (b.name, P)
        assert torch.isfinite(lse).all(), (b.name, P)
        max_abs, rel = compare(out_np, ref.cpu().numpy().astype(np.float64))
        assert max_abs <= MAX_ABS and rel <= REL_L2, (b.name, P, max_abs, rel)
        max_abs, rel = compare(out_np, oracles[id(b)])
        assert max_abs <= MAX_ABS and rel <= REL_L2, (b.name, P, max_abs, rel)


def test_noalloc_rejects_more_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _c_noalloc()
    # 64 sequences x 64 heads x 2048 partitions of 16 tokens: far above the limit
    _, need = pkv.decode_plan(64, 64, 8, 128, 16, 2048, 32768, 16)
    assert need > pkv.binding.NOALLOC_SCRATCH_BYTES
    out = torch.zeros(1, 64, 128, dtype=torch.float16, device="cuda")
    rc = fn(ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()), 64, 2048, 100, 0.1,
            64, 8, 128, 16, 32768, 16, None, None, None)
    assert rc == -3
