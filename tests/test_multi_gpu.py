"""Parity of the multi-token (causal) paged attention -- speculative-verify
and chunked-prefill shapes, through the C ABI -- with the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_213_gb300 as pkv
from gpu_util import assert_close
from paged_kv_cache_213_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.library()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _problem(lens, nq, H, Hk, d, bs, seed, poison=True):
    rng = np.random.default_rng(seed)
    batch = wl.make_batch("multi", list(lens), H, Hk, d, bs, rng, append=False, poison=poison)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = rng.standard_normal((int(qs[-1]), H, d)).astype(np.float16)
    return batch, q, qs


def _run(batch, q, qs, max_q_len, partition_tokens=0):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.full((q.shape[0], batch.n_q_heads), float("nan"), device="cuda")
    out = pkv.paged_decode_attention_multi(
        _t(q), _t(batch.k_cache), _t(batch.v_cache), _t(batch.block_tables),
        _t(batch.context_lens), _t(qs), batch.scale, batch.n_q_heads, batch.n_kv_heads,
        batch.head_dim, batch.block_size, max_q_len, max_context_len=batch.max_context_len,
        partition_tokens=partition_tokens, lse=lse, err_word=err)
    bits = pkv.get_error(err)
    return out.cpu().numpy(), lse.cpu().numpy().astype(np.float64), bits


def _oracle(batch, q, qs):
    return oracle.decode_multi(q, batch.k_cache, batch.v_cache, batch.block_tables,
                               batch.context_lens, qs, batch.scale, batch.n_q_heads,
                               batch.n_kv_heads, batch.head_dim, batch.block_size)


def _check(batch, q, qs, max_q_len, what, partition_tokens=0):
    out, lse, bits = _run(batch, q, qs, max_q_len, partition_tokens)
    assert bits == 0, what
    ref, ref_lse = _oracle(batch, q, qs)
    assert_close(out, ref, what=what)
    assert np.max(np.abs(lse - ref_lse)) <= 1e-4, what


def test_speculative_verify_llama3_8b_shape():
    """B=32, 32/8 heads, d=128: 4 draft tokens per sequence over contexts
    U{128..2048} (the LLaMA-3-8B-shaped layer)."""
    rng = np.random.default_rng(20262)
    lens = rng.integers(128, 2049, 32)
    batch, q, qs = _problem(lens, [4] * 32, 32, 8, 128, 16, 5)
    _check(batch, q, qs, 4, "verify 4 tokens")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_mixed_query_counts(d, g, bs):
    Hk = 2
    lens = [1, 7, 16, 17, 40, 130, 33, 5]
    nq = [1, 3, 16, 0, 9, 33, 33, 5]   # 0 queries, n = L (a full prefill), ...
    batch, q, qs = _problem(lens, nq, Hk * g, Hk, d, bs, 200 + d + 10 * g + bs)
    _check(batch, q, qs, max(nq), f"mixed d={d} g={g} bs={bs}")


@pytest.mark.parametrize("P", [16, 64, 256])
def test_forced_partitions(P):
    lens = [300, 17, 1000, 64]
    nq = [8, 2, 5, 1]
    batch, q, qs = _problem(lens, nq, 16, 4, 128, 16, 300 + P)
    _check(batch, q, qs, 8, f"P={P}", partition_tokens=P)


def test_chunked_prefill_chunk():
    """A 256-token prefill chunk after 344 cached tokens, next to decodes."""
    lens = [600, 50, 900]
    nq = [256, 1, 1]
    batch, q, qs = _problem(lens, nq, 8, 2, 128, 16, 401)
    _check(batch, q, qs, 256, "chunked prefill")


def test_one_query_per_sequence_matches_decode():
    rng = np.random.default_rng(7)
    lens = rng.integers(1, 300, 12)
    batch, q, qs = _problem(lens, [1] * 12, 16, 4, 128, 16, 8)
    out_m, lse_m, bits = _run(batch, q, qs, 1)
    assert bits == 0
    lse_d = torch.zeros(12, 16, device="cuda")
    out_d = pkv.paged_decode_attention(
        _t(q), _t(batch.k_cache), _t(batch.v_cache), _t(batch.block_tables),
        _t(batch.context_lens), batch.scale, 16, 4, 128, 16,
        max_context_len=batch.max_context_len, lse=lse_d).cpu().numpy()
    ref, _ = _oracle(batch, q, qs)
    assert_close(out_m, ref, what="multi n=1")
    assert_close(out_d, ref, what="decode")


def test_more_queries_than_context_is_flagged():
    batch, q, qs = _problem([5, 20], [6, 2], 8, 2, 128, 16, 9)
    out, lse, bits = _run(batch, q, qs, 6)
    assert bits & pkv.PKV_ERRBIT_CONTEXT
