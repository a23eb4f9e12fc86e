"""Helpers shared by the GPU parity tests: move a seeded batch to the GPU,
run the library on it, run the oracle on it, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_213_gb300 as pkv

# Tolerance for fp16 attention outputs against the oracle's exact (double)
# values: max-abs 2e-3 and relative L2 1e-2 over the compared outputs.
MAX_ABS = 2e-3
REL_L2 = 1e-2


def to_dev(batch, device="cuda"):
    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    d = dict(q=t(batch.q), k_cache=t(batch.k_cache), v_cache=t(batch.v_cache),
             block_tables=t(batch.block_tables), context_lens=t(batch.context_lens))
    if batch.has_append:
        d.update(k_new=t(batch.k_new), v_new=t(batch.v_new), slot_mapping=t(batch.slot_mapping))
    return d


def gpu_step(batch, dev=None, partition_tokens=0, want_lse=True, max_context_len="auto"):
    """Append (if the batch has one) then attend.  Returns numpy results and
    the error word's bits."""
    dev = dev or to_dev(batch)
    err = torch.zeros(1, dtype=torch.int32, device=dev["q"].device)
    if batch.has_append:
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"], err_word=err)
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device=dev["q"].device) \
        if want_lse else None
    mcl = batch.max_context_len if max_context_len == "auto" else max_context_len
    out = pkv.paged_decode_attention(
        dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
        batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
        max_context_len=mcl, partition_tokens=partition_tokens, lse=lse, err_word=err)
    bits = pkv.get_error(err)
    torch.cuda.synchronize()
    res = dict(out=out.cpu().numpy(), err=bits, dev=dev)
    if want_lse:
        res["lse"] = lse.cpu().numpy().astype(np.float64)
    return res


def oracle_step(batch, mask=None, num_threads=0):
    kc, vc = batch.k_cache, batch.v_cache
    if batch.has_append:
        kc, vc = oracle.append(batch.k_new, batch.v_new, batch.slot_mapping, kc, vc,
                               batch.block_size)
    out, lse, out16 = oracle.decode(batch.q, kc, vc, batch.block_tables, batch.context_lens,
                                    batch.scale, batch.n_q_heads, batch.n_kv_heads,
                                    batch.head_dim, batch.block_size, mask=mask,
                                    num_threads=num_threads)
    return dict(out=out, lse=lse, out16=out16, k_cache=kc, v_cache=vc)


def compare(gpu_out16, ref64, mask=None):
    """(max_abs, rel_l2) of fp16 GPU output against the oracle's doubles."""
    g = np.asarray(gpu_out16, dtype=np.float64)
    r = np.asarray(ref64, dtype=np.float64)
    if mask is not None:
        g = g[mask]
        r = r[mask]
    diff = g - r
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(gpu_out16, ref64, mask=None, what=""):
    max_abs, rel = compare(gpu_out16, ref64, mask)
    assert np.all(np.isfinite(np.asarray(gpu_out16, dtype=np.float64)[mask] if mask is not None
                              else np.asarray(gpu_out16, dtype=np.float64))), f"{what}: non-finite"
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel={rel:.3e}"
    return max_abs, rel


def relayout(base, bs, seed, shared=None):
    """The same logical K/V (and q) as `base` (attention-only batch) in a new
    pool: block size `bs`, a fresh random physical order, optional sharing."""
    from paged_kv_cache_213_gb300 import workloads as wl
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in base.context_lens]
    b2 = wl.make_batch("relayout", lens, base.n_q_heads, base.n_kv_heads, base.head_dim, bs,
                       rng, scale=base.scale, append=False, poison=True, shared=shared)
    b2.q = base.q
    bs0 = base.block_size
    for b, L in enumerate(lens):
        t = np.arange(L)
        src_k = base.k_cache[base.block_tables[b, t // bs0], :, t % bs0, :]
        src_v = base.v_cache[base.block_tables[b, t // bs0], :, t % bs0, :]
        b2.k_cache[b2.block_tables[b, t // bs], :, t % bs, :] = src_k
        b2.v_cache[b2.block_tables[b, t // bs], :, t % bs, :] = src_v
    return b2
