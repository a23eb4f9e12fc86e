"""Seeded random problems through the main entry points, against the oracle.

Each case draws its shape (head_dim, GQA group size, KV heads, block size),
a batch of 1 to 300 sequences and a length mix (empty sequences, lengths
below a block, block multiples and their neighbours, log-uniform up to a few
thousand tokens), with NaN poison in every cache row and table entry that no
sequence reads.  The fp16 entry runs with the automatic split and with a
random fixed partition; the E4M3, multi-token and prefix-aware entries run on
draws of their own supported shapes.  Every output and lse is compared with
the oracle; the seed names the case."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_213_gb300 as pkv
from gpu_util import assert_close, gpu_step, oracle_step, to_dev
from paged_kv_cache_213_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_TOKENS = 120_000  # per case: keeps the oracle to about a second


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.library()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _lens(rng, B, bs, allow_empty):
    kind = int(rng.integers(4))
    if kind == 0:
        lens = rng.integers(0 if allow_empty else 1, 600, B)
    elif kind == 1:  # log-uniform
        lens = np.exp(rng.uniform(0, math.log(4000), B)).astype(np.int64)
    elif kind == 2:  # a few long sequences among short ones
        lens = rng.integers(1, 40, B)
        long_ = rng.random(B) < 0.1
        lens[long_] = rng.integers(1000, 5000, int(long_.sum()))
    else:  # block multiples and their neighbours
        lens = bs * rng.integers(1, 40, B) + rng.integers(-1, 2, B)
    lens = np.maximum(lens, 0 if allow_empty else 1)
    if allow_empty and B > 2:
        lens[rng.integers(0, B)] = 0
    total = int(lens.sum())
    if total > MAX_TOKENS:  # scale the mix down, keeping its shape
        lens = np.maximum(lens * MAX_TOKENS // total, 0 if allow_empty else 1)
    return [int(x) for x in lens]


def _shape(rng, block_sizes, groups=(1, 2, 4, 8)):
    d = int(rng.choice([64, 128]))
    g = int(rng.choice(groups))
    hk = int(rng.choice([1, 2, 3, 4, 8]))
    bs = int(rng.choice(block_sizes))
    B = int(rng.choice([1, 2, 3, 7, 16, 33, 64, 130, 300]))
    return d, g, hk, bs, B


@pytest.mark.parametrize("seed", range(48))
def test_fp16_random(seed):
    rng = np.random.default_rng(7000 + seed)
    d, g, hk, bs, B = _shape(rng, [1, 2, 4, 8, 16, 32, 64, 128, 256])
    append = bool(rng.integers(2))
    lens = _lens(rng, B, bs, allow_empty=not append)
    batch = wl.make_batch(f"fuzz{seed}", lens, g * hk, hk, d, bs, rng, append=append,
                          poison=True)
    ref = oracle_step(batch)
    step = math.lcm(16, bs)
    P = step * int(rng.integers(1, max(2, 1024 // step + 1)))
    auto = None
    for part in (0, P):
        got = gpu_step(batch, partition_tokens=part)
        what = f"seed {seed}: d={d} g={g} Hk={hk} bs={bs} B={B} P={part}"
        assert got["err"] == 0, what
        assert_close(got["out"], ref["out"], what=what)
        finite = np.isfinite(ref["lse"])
        assert np.array_equal(np.isfinite(got["lse"]), finite), what
        assert np.max(np.abs(got["lse"][finite] - ref["lse"][finite]), initial=0.0) <= 1e-4, what
        auto = got["out"] if part == 0 else auto
    if append:  # the one-call step, then the flagged call after it: bit-identical
        dev = to_dev(batch)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = (dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                dev["context_lens"], batch.scale, g * hk, hk, d, bs)
        stepped = pkv.paged_decode_step(dev["k_new"], dev["v_new"], dev["slot_mapping"], *args,
                                        max_context_len=batch.max_context_len, err_word=err)
        flagged = pkv.paged_decode_attention(*args, max_context_len=batch.max_context_len,
                                             err_word=err, flags=pkv.PKV_TABLES_READY)
        # the one-launch step (the attention appends the newest tokens itself)
        dev2 = to_dev(batch)
        args2 = (dev2["q"], dev2["k_cache"], dev2["v_cache"], dev2["block_tables"],
                 dev2["context_lens"], batch.scale, g * hk, hk, d, bs)
        fused = pkv.paged_decode_step(dev2["k_new"], dev2["v_new"], dev2["slot_mapping"],
                                      *args2, max_context_len=batch.max_context_len,
                                      err_word=err,
                                      flags=pkv.PKV_APPEND_NEWEST | pkv.PKV_TABLES_READY)
        assert pkv.get_error(err) == 0
        for o in (stepped, flagged, fused):
            assert np.array_equal(o.cpu().numpy().view(np.uint16), auto.view(np.uint16))
        assert np.array_equal(dev2["k_cache"].cpu().numpy().view(np.uint16),
                              dev["k_cache"].cpu().numpy().view(np.uint16))
        assert np.array_equal(dev2["v_cache"].cpu().numpy().view(np.uint16),
                              dev["v_cache"].cpu().numpy().view(np.uint16))


def _amax_scale(*arrays):
    m = 1e-6
    for a in arrays:
        f = a.astype(np.float32)
        f = f[np.isfinite(f)]
        if f.size:
            m = max(m, float(np.max(np.abs(f))))
    return np.float32(m / 448.0)


@pytest.mark.parametrize("seed", range(24))
def test_e4m3_random(seed):
    rng = np.random.default_rng(8000 + seed)
    d, g, hk, bs, B = _shape(rng, [16, 32, 64, 128])
    append = bool(rng.integers(2))
    lens = _lens(rng, B, bs, allow_empty=not append)
    batch = wl.make_batch(f"fuzz8_{seed}", lens, g * hk, hk, d, bs, rng, append=append,
                          poison=True)
    srcs_k = [batch.k_cache] + ([batch.k_new] if append else [])
    srcs_v = [batch.v_cache] + ([batch.v_new] if append else [])
    ks, vs = _amax_scale(*srcs_k), _amax_scale(*srcs_v)
    kc8, vc8 = oracle.quantize_e4m3(batch.k_cache, ks), oracle.quantize_e4m3(batch.v_cache, vs)
    rk, rv = kc8, vc8
    if append:
        rk, rv = oracle.append_f8(batch.k_new, batch.v_new, batch.slot_mapping, kc8, vc8, bs,
                                  ks, vs)
    ref, ref_lse = oracle.decode_f8(batch.q, rk, rv, ks, vs, batch.block_tables,
                                    batch.context_lens, batch.scale, batch.n_q_heads, hk, d, bs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = _t(kc8), _t(vc8)
    if append:
        pkv.paged_kv_append_fp8(_t(batch.k_new), _t(batch.v_new), _t(batch.slot_mapping), kc,
                                vc, ks, vs, err_word=err)
    lse = torch.full((B, g * hk), float("nan"), device="cuda")
    out = pkv.paged_decode_attention_fp8(
        _t(batch.q), kc, vc, _t(batch.block_tables), _t(batch.context_lens), batch.scale, ks,
        vs, g * hk, hk, d, bs, max_context_len=batch.max_context_len, lse=lse, err_word=err)
    what = f"seed {seed}: d={d} g={g} Hk={hk} bs={bs} B={B}"
    assert pkv.get_error(err) == 0, what
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv), what
    if append:  # the one-call step: the same codes and output as append + attention
        kc2, vc2 = _t(kc8), _t(vc8)
        stepped = pkv.paged_decode_step_fp8(
            _t(batch.k_new), _t(batch.v_new), _t(batch.slot_mapping), _t(batch.q), kc2, vc2,
            _t(batch.block_tables), _t(batch.context_lens), batch.scale, ks, vs, g * hk, hk, d,
            bs, max_context_len=batch.max_context_len, err_word=err,
            flags=pkv.PKV_APPEND_NEWEST | pkv.PKV_TABLES_READY)
        assert pkv.get_error(err) == 0, what
        assert np.array_equal(kc2.cpu().numpy(), rk) and np.array_equal(vc2.cpu().numpy(), rv)
        assert np.array_equal(stepped.cpu().numpy().view(np.uint16),
                              out.cpu().numpy().view(np.uint16)), what
    assert_close(out.cpu().numpy(), ref, what=what)
    got_lse = lse.cpu().numpy().astype(np.float64)
    finite = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), finite), what
    assert np.max(np.abs(got_lse[finite] - ref_lse[finite]), initial=0.0) <= 1e-4, what


@pytest.mark.parametrize("seed", range(24))
def test_multi_token_random(seed):
    rng = np.random.default_rng(9000 + seed)
    d, g, hk, bs, B = _shape(rng, [16, 32, 64])
    lens = _lens(rng, B, bs, allow_empty=True)
    # 0 .. 4 new tokens per sequence (never more than its length); sometimes
    # a prefill-sized count
    nq = [int(min(L, rng.integers(0, 5))) for L in lens]
    if B > 1 and rng.random() < 0.3:
        i = int(np.argmax(lens))
        nq[i] = int(min(lens[i], rng.integers(16, 200)))
    batch = wl.make_batch(f"fuzzm{seed}", lens, g * hk, hk, d, bs, rng, append=False,
                          poison=True)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    total_q = int(qs[-1])
    q = rng.standard_normal((total_q, g * hk, d)).astype(np.float16)
    ref, ref_lse = oracle.decode_multi(q, batch.k_cache, batch.v_cache, batch.block_tables,
                                       batch.context_lens, qs, batch.scale, g * hk, hk, d, bs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.full((total_q, g * hk), float("nan"), device="cuda")
    out = pkv.paged_decode_attention_multi(
        _t(q), _t(batch.k_cache), _t(batch.v_cache), _t(batch.block_tables),
        _t(batch.context_lens), _t(qs), batch.scale, g * hk, hk, d, bs, max(max(nq), 1),
        max_context_len=batch.max_context_len, lse=lse, err_word=err)
    what = f"seed {seed}: d={d} g={g} Hk={hk} bs={bs} B={B} max_q={max(nq)}"
    assert pkv.get_error(err) == 0, what
    if total_q:
        assert_close(out.cpu().numpy(), ref, what=what)
        got_lse = lse.cpu().numpy().astype(np.float64)
        finite = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(got_lse), finite), what
        assert np.max(np.abs(got_lse[finite] - ref_lse[finite]), initial=0.0) <= 1e-4, what


@pytest.mark.parametrize("seed", range(24))
def test_prefix_shared_random(seed):
    rng = np.random.default_rng(10000 + seed)
    d, g, hk, bs, _ = _shape(rng, [16, 32])
    lens, shared, b = [], [], 0
    for _ in range(int(rng.integers(1, 12))):  # groups of consecutive sequences
        n = int(rng.integers(1, 7))
        pre_blocks = int(rng.integers(1, 40))
        for _ in range(n):  # private parts; a member may stop inside the prefix
            lens.append(int(max(1, pre_blocks * bs + rng.integers(-bs, 3 * bs))))
        if n > 1:
            shared.append((list(range(b, b + n)), pre_blocks))
        b += n
    # no append: a member that stops inside the prefix would append into a
    # shared block, and two such members could write one slot in one call
    batch = wl.make_batch(f"fuzzp{seed}", lens, g * hk, hk, d, bs, rng, append=False,
                          poison=True, shared=shared)
    ref = oracle_step(batch)
    offs, pref, gmax, pmax = wl.prefix_groups(batch)
    saved = os.environ.pop("PKV_PREFIX_PASS", None)
    try:
        for pass_ in ("shared", None):
            if pass_:
                os.environ["PKV_PREFIX_PASS"] = pass_
            else:
                os.environ.pop("PKV_PREFIX_PASS", None)
            dev = to_dev(batch)
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            lse = torch.full((batch.num_seqs, g * hk), float("nan"), device="cuda")
            out = pkv.paged_decode_attention_prefix_shared(
                dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                dev["context_lens"], batch.scale, g * hk, hk, d, bs, _t(offs), _t(pref), gmax,
                pmax, max_context_len=batch.max_context_len, lse=lse, err_word=err)
            what = f"seed {seed}: d={d} g={g} Hk={hk} bs={bs} groups={len(offs) - 1} {pass_}"
            assert pkv.get_error(err) == 0, what
            assert_close(out.cpu().numpy(), ref["out"], what=what)
            got_lse = lse.cpu().numpy().astype(np.float64)
            assert np.max(np.abs(got_lse - ref["lse"])) <= 1e-4, what
    finally:
        os.environ.pop("PKV_PREFIX_PASS", None)
        if saved is not None:
            os.environ["PKV_PREFIX_PASS"] = saved
