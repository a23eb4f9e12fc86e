"""Prefix-aware decode attention (shared prefix read once per group chunk)
against the oracle: the Mistral-shaped mix and the 70B parallel-sampling
workloads, and edge cases -- prefixes that are not whole tiles, members
shorter than the prefix, sequences with no private tile, groups larger than
one CTA chunk, one-sequence groups, every GQA group size and head_dim."""
import os

import numpy as np
import pytest
import torch

import paged_kv_cache_213_gb300 as pkv
from gpu_util import assert_close, oracle_step, to_dev
from paged_kv_cache_213_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.library()


def run_shared(batch, groups=None, pass_="shared", flags=0):
    """The prefix-aware entry point; pass_ fixes its choice between the
    two-pass path ("shared") and the regular attention ("regular"), or leaves
    it to the library (None); flags are its launch flags."""
    saved = os.environ.pop("PKV_PREFIX_PASS", None)
    if pass_ is not None:
        os.environ["PKV_PREFIX_PASS"] = pass_
    try:
        return _run_shared(batch, groups, flags)
    finally:
        os.environ.pop("PKV_PREFIX_PASS", None)
        if saved is not None:
            os.environ["PKV_PREFIX_PASS"] = saved


def _run_shared(batch, groups=None, flags=0):
    offs, pref, gmax, pmax = groups if groups is not None else wl.prefix_groups(batch)
    dev = to_dev(batch)
    if batch.has_append:
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"])
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.paged_decode_attention_prefix_shared(
        dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
        batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
        torch.from_numpy(offs).cuda(), torch.from_numpy(pref).cuda(), gmax, pmax,
        max_context_len=batch.max_context_len, lse=lse, err_word=err, flags=flags)
    assert pkv.get_error(err) == 0
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("pass_", ["shared", None, "regular"])
@pytest.mark.parametrize("cfg", [3, 5])
def test_shared_workloads(cfg, pass_):
    """Every output and lse of the full-size workload against the oracle,
    through the two-pass path, the library's choice and the regular path."""
    batch = wl.workload(cfg, poison=True)
    out, lse = run_shared(batch, pass_=pass_)
    ref = oracle_step(batch)
    assert_close(out, ref["out"], what=f"workload {cfg}")
    assert np.max(np.abs(lse - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_shared_edge_cases(d, G):
    rng = np.random.default_rng(700 + 10 * d + G)
    Hk = 2
    # group A: 5 members, prefix 3 blocks, one member shorter than the prefix
    # group B: 2 members sharing everything they have (no private tile)
    # group C: one sequence; group D: 3 members with a prefix that is no whole tile
    lens = [100, 60, 33, 130, 75, 64, 64, 40, 90, 91, 70]
    shared = [([0, 1, 2, 3, 4], 3), ([5, 6], 4), ([8, 9, 10], 3)]
    batch = wl.make_batch("edge", lens, Hk * G, Hk, d, 16, rng, append=False, poison=True,
                          shared=shared)
    offs = np.array([0, 5, 7, 8, 11], dtype=np.int32)
    pref = np.array([48, 64, 0, 37], dtype=np.int32)
    out, lse = run_shared(batch, (offs, pref, 5, 64))
    ref = oracle_step(batch)
    assert_close(out, ref["out"], what=f"d={d} G={G}")
    assert np.max(np.abs(lse - ref["lse"])) <= 1e-4


def test_group_larger_than_a_chunk_and_block_size_32():
    rng = np.random.default_rng(9)
    G = 4  # 4 members per warp, 16 per CTA chunk
    lens = list(rng.integers(200, 400, size=40))
    batch = wl.make_batch("big", lens, 8 * G, 8, 128, 32, rng, append=True, poison=True,
                          shared=[(list(range(40)), 6)])
    out, _ = run_shared(batch, (np.array([0, 40], dtype=np.int32),
                                np.array([192], dtype=np.int32), 40, 192))
    ref = oracle_step(batch)
    assert_close(out, ref["out"], what="40 members, bs 32")


def test_matches_regular_entry_point():
    batch = wl.workload(5, poison=False)
    out, _ = run_shared(batch)
    dev = to_dev(batch)
    reg = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                     dev["block_tables"], dev["context_lens"], batch.scale,
                                     batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                                     batch.block_size, max_context_len=batch.max_context_len)
    diff = np.abs(out.astype(np.float64) - reg.cpu().numpy().astype(np.float64))
    assert diff.max() <= 2e-3


def test_many_groups_of_forked_completions():
    """64 prompts x 4 completions with 128-token prefixes and short private
    suffixes (2048 grouped (sequence, KV head) segments): the two-pass path
    and the library's choice both match the oracle."""
    rng = np.random.default_rng(21)
    groups = [(list(range(4 * p, 4 * p + 4)), 8) for p in range(64)]  # 128-token prefixes
    lens = [128 + int(x) for x in rng.integers(1, 40, size=256)]
    batch = wl.make_batch("many", lens, 16, 8, 64, 16, rng, append=False, poison=True,
                          shared=groups)
    ref = oracle_step(batch)
    for pass_ in ("shared", None):
        out, lse = run_shared(batch, pass_=pass_)
        assert_close(out, ref["out"], what=f"pass={pass_}")
        assert np.max(np.abs(lse - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("pass_", ["shared", "regular"])
@pytest.mark.parametrize("cfg", [3, 5])
def test_tables_ready_flag(cfg, pass_):
    """paged_decode_attention_prefix_shared_ex with PKV_TABLES_READY (the
    groups and lengths read before the dependency wait): bit-identical to the
    call without the flag, every output against the oracle."""
    batch = wl.workload(cfg, poison=True)
    out_f, lse_f = run_shared(batch, pass_=pass_, flags=pkv.PKV_TABLES_READY)
    out_p, lse_p = run_shared(batch, pass_=pass_)
    assert np.array_equal(out_f.view(np.uint16), out_p.view(np.uint16))
    assert np.array_equal(lse_f, lse_p)
    ref = oracle_step(batch)
    assert_close(out_f, ref["out"], what=f"flagged workload {cfg}")
    assert np.max(np.abs(lse_f - ref["lse"])) <= 1e-4
