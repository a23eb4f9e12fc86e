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


# --- the balanced split (partition_tokens = 0, max_q_len * g <= 16) --------

def _run_into(batch, q, qs, max_q_len, partition_tokens=0, workspace=None):
    """The call with NaN-filled out and lse, so unwritten rows stay NaN."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((q.shape[0], batch.n_q_heads), float("nan"), device="cuda")
    pkv.paged_decode_attention_multi(
        _t(q), _t(batch.k_cache), _t(batch.v_cache), _t(batch.block_tables),
        _t(batch.context_lens), _t(qs), batch.scale, batch.n_q_heads, batch.n_kv_heads,
        batch.head_dim, batch.block_size, max_q_len, max_context_len=batch.max_context_len,
        partition_tokens=partition_tokens, out=out, workspace=workspace, lse=lse, err_word=err)
    bits = pkv.get_error(err)
    return out.cpu().numpy(), lse.cpu().numpy().astype(np.float64), bits


def _balanced(batch, qs, max_q_len):
    P, ws = pkv.multi_plan(batch.num_seqs, int(qs[-1]), max_q_len, batch.n_q_heads,
                           batch.n_kv_heads, batch.head_dim, batch.block_size,
                           batch.max_blocks_per_seq, batch.max_context_len, 0)
    return P == 0 and ws > 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_balanced_split_ragged(d, g, bs):
    """Every (query row, head) against the oracle on the balanced split:
    0 queries, n = L (a whole short prefill), L = 0, single tokens and the
    most rows one segment holds (16 / g tokens), over ragged lengths; the
    fixed-partition kernel on the same batch agrees."""
    nmax = 16 // g
    Hk = 2
    lens = [1, 7, 16, 17, 40, 130, 0, 5, 300, 2, 64, 1000]
    nq = [1, min(nmax, 7), min(nmax, 16), 0, nmax, nmax, 0, min(nmax, 5), 1, min(nmax, 2),
          nmax, max(1, nmax - 1)]
    batch, q, qs = _problem(lens, nq, Hk * g, Hk, d, bs, 500 + d + 10 * g + bs)
    assert _balanced(batch, qs, nmax)
    out, lse, bits = _run_into(batch, q, qs, nmax)
    assert bits == 0
    ref, ref_lse = _oracle(batch, q, qs)
    assert_close(out, ref, what=f"balanced d={d} g={g} bs={bs}")
    assert np.max(np.abs(lse - ref_lse)) <= 1e-4
    out_p, _, bits_p = _run_into(batch, q, qs, nmax, partition_tokens=64)
    assert bits_p == 0
    assert_close(out_p, ref, what="fixed partitions")


def test_balanced_split_many_segments():
    """96 sequences x 8 KV heads (more segments than twice the SMs: 4-warp
    CTAs), 4 draft tokens each over short contexts, every row checked."""
    rng = np.random.default_rng(77)
    lens = rng.integers(4, 700, 96)
    batch, q, qs = _problem(lens, [4] * 96, 32, 8, 128, 16, 78)
    assert _balanced(batch, qs, 4)
    out, lse, bits = _run_into(batch, q, qs, 4)
    assert bits == 0
    ref, ref_lse = _oracle(batch, q, qs)
    assert_close(out, ref, what="many segments")
    assert np.max(np.abs(lse - ref_lse)) <= 1e-4


def test_balanced_split_long_contexts_cut_segments():
    """Few long sequences (every segment cut over many warps, merged by the
    last arriver), 2 tokens x g = 8 rows; two calls on one workspace give
    bit-identical results (the counters are left zero, the order is fixed)."""
    lens = [16384, 9000, 20000, 777]
    batch, q, qs = _problem(lens, [2, 2, 1, 2], 32, 4, 128, 16, 79)
    P, ws = pkv.multi_plan(4, int(qs[-1]), 2, 32, 4, 128, 16, batch.max_blocks_per_seq,
                           batch.max_context_len, 0)
    assert P == 0
    work = torch.zeros(ws, dtype=torch.uint8, device="cuda")
    out1, lse1, bits1 = _run_into(batch, q, qs, 2, workspace=work)
    out2, lse2, bits2 = _run_into(batch, q, qs, 2, workspace=work)
    assert bits1 == 0 and bits2 == 0
    assert np.array_equal(out1.view(np.uint16), out2.view(np.uint16))
    assert np.array_equal(lse1, lse2)
    ref, ref_lse = _oracle(batch, q, qs)
    assert_close(out1, ref, what="long contexts")
    assert np.max(np.abs(lse1 - ref_lse)) <= 1e-4


@pytest.mark.parametrize("partition_tokens", [0, 32])
def test_query_count_above_max_q_len_is_flagged(partition_tokens):
    """A sequence with more query tokens than max_q_len is flagged and its
    rows are left unwritten; the others are computed (balanced split and
    fixed partitions alike)."""
    batch, q, qs = _problem([50, 80, 33], [2, 5, 1], 16, 4, 128, 16, 80)
    out, lse, bits = _run_into(batch, q, qs, 2, partition_tokens=partition_tokens)
    assert bits & pkv.PKV_ERRBIT_CONTEXT
    ref, ref_lse = _oracle(batch, q, qs)
    bad = slice(int(qs[1]), int(qs[2]))
    assert np.isnan(out[bad].astype(np.float32)).all() and np.isnan(lse[bad]).all()
    good = np.r_[int(qs[0]):int(qs[1]), int(qs[2]):int(qs[3])]
    assert_close(out[good], ref[good], what="unflagged rows")


def test_balanced_split_timeout_recovers(monkeypatch):
    """The bounded-wait hook on the multi-token kernel: the call returns with
    PKV_ERRBIT_TIMEOUT; after the workspace is zeroed again, a normal call
    matches the oracle."""
    rng = np.random.default_rng(81)
    lens = rng.integers(100, 3000, 32)
    batch, q, qs = _problem(lens, [4] * 32, 32, 8, 128, 16, 82)
    P, ws = pkv.multi_plan(32, int(qs[-1]), 4, 32, 8, 128, 16, batch.max_blocks_per_seq,
                           batch.max_context_len, 0)
    assert P == 0
    work = torch.zeros(ws, dtype=torch.uint8, device="cuda")
    monkeypatch.setenv("PKV_TEST_WAIT_POLLS", "0")
    _, _, bits = _run_into(batch, q, qs, 4, workspace=work)
    torch.cuda.synchronize()
    assert bits & pkv.PKV_ERRBIT_TIMEOUT and not bits & ~pkv.PKV_ERRBIT_TIMEOUT, bits
    monkeypatch.delenv("PKV_TEST_WAIT_POLLS")
    work.zero_()
    out, lse, bits = _run_into(batch, q, qs, 4, workspace=work)
    assert bits == 0
    ref, _ = _oracle(batch, q, qs)
    assert_close(out, ref, what="after the timeout")


def test_balanced_split_stale_counters_flagged():
    """A workspace of 0xFF bytes (counters -1) on the multi-token balanced
    split: the call returns with PKV_ERRBIT_WORKSPACE (the counters are only
    counted, never waited on); after paged_decode_workspace_clear a call
    matches the oracle."""
    rng = np.random.default_rng(85)
    lens = rng.integers(100, 3000, 32)
    batch, q, qs = _problem(lens, [4] * 32, 32, 8, 128, 16, 86)
    assert _balanced(batch, qs, 4)
    _, ws = pkv.multi_plan(32, int(qs[-1]), 4, 32, 8, 128, 16, batch.max_blocks_per_seq,
                           batch.max_context_len, 0)
    work = torch.full((ws,), 0xFF, dtype=torch.uint8, device="cuda")
    _, _, bits = _run_into(batch, q, qs, 4, workspace=work)
    torch.cuda.synchronize()
    assert bits == pkv.PKV_ERRBIT_WORKSPACE, bits
    pkv.paged_decode_workspace_clear(work)
    out, _, bits = _run_into(batch, q, qs, 4, workspace=work)
    assert bits == 0
    ref, _ = _oracle(batch, q, qs)
    assert_close(out, ref, what="after the clear")


def test_tables_ready_flag():
    """paged_decode_attention_multi_ex with PKV_TABLES_READY (lengths, tables
    and query_start read before the dependency wait), back to back:
    bit-identical to the call without it, and the oracle's result."""
    rng = np.random.default_rng(83)
    lens = rng.integers(64, 2049, 32)
    batch, q, qs = _problem(lens, [4] * 32, 32, 8, 128, 16, 84)
    dq, kc, vc, bt, cl, dqs = (_t(q), _t(batch.k_cache), _t(batch.v_cache),
                               _t(batch.block_tables), _t(batch.context_lens), _t(qs))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [pkv.paged_decode_attention_multi(
        dq, kc, vc, bt, cl, dqs, batch.scale, 32, 8, 128, 16, 4,
        max_context_len=batch.max_context_len, err_word=err, flags=f).cpu().numpy()
        for f in (pkv.PKV_TABLES_READY, pkv.PKV_TABLES_READY, 0)]
    assert pkv.get_error(err) == 0
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16))
    ref, _ = _oracle(batch, q, qs)
    assert_close(outs[0], ref, what="flagged multi-token")
