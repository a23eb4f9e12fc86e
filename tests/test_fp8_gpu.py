"""Parity of the FP8 (E4M3) KV-cache path -- the quantizing append and the
attention over E4M3 caches, through the C ABI -- with the CPU oracle's FP8
statement: bit-exact codes for the append, the fp16 attention tolerance for
the outputs.  The E4M3 caches are the oracle's quantization of the seeded
fp16 workloads (NaN poison becomes the NaN code)."""
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


def _amax_scale(*arrays):
    """max |finite value| / 448 over the arrays, as fp32."""
    m = 0.0
    for a in arrays:
        if a is None:
            continue
        f = a.astype(np.float32)
        f = f[np.isfinite(f)]
        if f.size:
            m = max(m, float(np.max(np.abs(f))))
    return np.float32(max(m, 1e-6) / 448.0)


def _scales(batch):
    return (_amax_scale(batch.k_cache, batch.k_new if batch.has_append else None),
            _amax_scale(batch.v_cache, batch.v_new if batch.has_append else None))


def _caches8(batch, ks, vs):
    return oracle.quantize_e4m3(batch.k_cache, ks), oracle.quantize_e4m3(batch.v_cache, vs)


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_f8(batch, kc8, vc8, ks, vs, slot_mapping=None):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = _t(kc8), _t(vc8)
    if batch.has_append:
        sm = _t(batch.slot_mapping if slot_mapping is None else slot_mapping)
        pkv.paged_kv_append_fp8(_t(batch.k_new), _t(batch.v_new), sm, kc, vc, ks, vs,
                                err_word=err)
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
    out = pkv.paged_decode_attention_fp8(
        _t(batch.q), kc, vc, _t(batch.block_tables), _t(batch.context_lens), batch.scale, ks,
        vs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
        max_context_len=batch.max_context_len, lse=lse, err_word=err)
    bits = pkv.get_error(err)
    torch.cuda.synchronize()
    return dict(out=out.cpu().numpy(), lse=lse.cpu().numpy().astype(np.float64), err=bits,
                k_cache=kc.cpu().numpy(), v_cache=vc.cpu().numpy())


def oracle_f8(batch, kc8, vc8, ks, vs, mask=None):
    if batch.has_append:
        kc8, vc8 = oracle.append_f8(batch.k_new, batch.v_new, batch.slot_mapping, kc8, vc8,
                                    batch.block_size, ks, vs)
    out, lse = oracle.decode_f8(batch.q, kc8, vc8, ks, vs, batch.block_tables,
                                batch.context_lens, batch.scale, batch.n_q_heads,
                                batch.n_kv_heads, batch.head_dim, batch.block_size, mask=mask)
    return dict(out=out, lse=lse, k_cache=kc8, v_cache=vc8)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_fp8_workload_parity(cfg):
    """Full-size workloads with E4M3 caches, poisoned; every output and lse
    compared; the append's codes bit-exact over the whole pool."""
    batch = wl.workload(cfg, poison=True)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    assert np.any(kc8 == 0x7F)  # the poison became NaN codes
    g = gpu_f8(batch, kc8, vc8, ks, vs)
    assert g["err"] == 0
    ref = oracle_f8(batch, kc8, vc8, ks, vs)
    assert_close(g["out"], ref["out"], what=f"fp8 workload {cfg}")
    assert np.max(np.abs(g["lse"] - ref["lse"])) <= 1e-4
    if batch.has_append:
        assert np.array_equal(g["k_cache"], ref["k_cache"])
        assert np.array_equal(g["v_cache"], ref["v_cache"])


def test_fp8_append_saturation_padding_and_bad_slot():
    rng = np.random.default_rng(31)
    batch = wl.make_batch("f8pad", [5, 16, 17, 33], 8, 2, 128, 16, rng, append=True,
                          poison=True, append_padding=3)
    batch.k_new = (batch.k_new.astype(np.float32) * 30.0).astype(np.float16)  # some overflow
    ks, vs = np.float32(0.05), np.float32(0.01)
    assert np.any(np.abs(batch.k_new.astype(np.float32) / ks) > 448.0)
    kc8, vc8 = _caches8(batch, ks, vs)
    g = gpu_f8(batch, kc8, vc8, ks, vs)
    ref = oracle_f8(batch, kc8, vc8, ks, vs, mask=np.zeros((4, 8), dtype=bool))
    assert g["err"] == 0
    assert np.array_equal(g["k_cache"], ref["k_cache"])
    assert np.array_equal(g["v_cache"], ref["v_cache"])
    # a slot beyond the pool is flagged and skipped; the other tokens land
    bad = batch.slot_mapping.copy()
    first = int(np.nonzero(bad >= 0)[0][0])
    bad[first] = batch.num_blocks * batch.block_size + 1
    g2 = gpu_f8(batch, kc8, vc8, ks, vs, slot_mapping=bad)
    assert g2["err"] & pkv.PKV_ERRBIT_SLOT
    keep = bad.copy()
    keep[first] = -1
    ref2 = oracle.append_f8(batch.k_new, batch.v_new, keep, kc8, vc8, batch.block_size, ks, vs)
    assert np.array_equal(g2["k_cache"], ref2[0]) and np.array_equal(g2["v_cache"], ref2[1])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32])
def test_fp8_edge_shapes(d, g, bs):
    Hk = 2
    H = Hk * g
    rng = np.random.default_rng(100 + d + 10 * g + bs)
    lens = [1, 15, 16, 17, 33, 130, 0, 64]
    batch = wl.make_batch("f8edge", lens, H, Hk, d, bs, rng, append=False, poison=True)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    got = gpu_f8(batch, kc8, vc8, ks, vs)
    assert got["err"] == 0
    ref = oracle_f8(batch, kc8, vc8, ks, vs)
    assert_close(got["out"], ref["out"], what=f"fp8 d={d} g={g} bs={bs}")
    live = np.asarray(lens) > 0
    assert np.max(np.abs(got["lse"][live] - ref["lse"][live])) <= 1e-4
    assert np.all(got["out"][~live] == 0) and np.all(np.isneginf(got["lse"][~live]))


def test_fp8_one_token_is_its_value_row():
    """L = 1: the output is the dequantized V row (p = 1), within fp16 rounding."""
    rng = np.random.default_rng(41)
    batch = wl.make_batch("f8one", [1, 1, 1], 8, 2, 128, 16, rng, append=False, poison=True)
    ks, vs = np.float32(0.02), np.float32(0.013)
    kc8, vc8 = _caches8(batch, ks, vs)
    got = gpu_f8(batch, kc8, vc8, ks, vs)
    table = oracle.e4m3_table()
    for b in range(3):
        blk = batch.block_tables[b, 0]
        for h in range(8):
            row = table[vc8[blk, h // 4, 0]] * float(vs)
            assert np.max(np.abs(got["out"][b, h].astype(np.float64) - row)) <= \
                2.0 ** -11 * max(1.0, np.max(np.abs(row)))


def test_fp8_host_rejections():
    rng = np.random.default_rng(42)
    batch = wl.make_batch("f8rej", [20, 5], 8, 2, 128, 16, rng, append=False, poison=False)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    with pytest.raises(pkv.PagedKVError) as e:  # too small a workspace
        pkv.paged_decode_attention_fp8(
            _t(batch.q), _t(kc8), _t(vc8), _t(batch.block_tables), _t(batch.context_lens),
            batch.scale, ks, vs, 8, 2, 128, 16, workspace=torch.zeros(256, dtype=torch.uint8,
                                                                      device="cuda"))
    assert e.value.status == -3
    with pytest.raises(pkv.PagedKVError) as e:  # a zero scale
        pkv.paged_decode_attention_fp8(
            _t(batch.q), _t(kc8), _t(vc8), _t(batch.block_tables), _t(batch.context_lens),
            batch.scale, 0.0, vs, 8, 2, 128, 16)
    assert e.value.status == -1
    b8 = wl.make_batch("f8bs8", [20, 5], 8, 2, 128, 8, rng, append=False, poison=False)
    with pytest.raises(pkv.PagedKVError) as e:  # block size 8: no balanced split
        pkv.paged_decode_attention_fp8(
            _t(b8.q), _t(oracle.quantize_e4m3(b8.k_cache, ks)),
            _t(oracle.quantize_e4m3(b8.v_cache, vs)), _t(b8.block_tables),
            _t(b8.context_lens), b8.scale, ks, vs, 8, 2, 128, 8)
    assert e.value.status == -2


# --- the prefix-aware call over E4M3 caches --------------------------------

def gpu_f8_shared(batch, kc8, vc8, ks, vs, groups=None, pass_="shared"):
    """Append (if any) then paged_decode_attention_prefix_shared_fp8; pass_
    fixes the two-pass path ("shared"), or leaves the choice to the library
    (None)."""
    import os
    offs, pref, gmax, pmax = groups if groups is not None else wl.prefix_groups(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = _t(kc8), _t(vc8)
    if batch.has_append:
        pkv.paged_kv_append_fp8(_t(batch.k_new), _t(batch.v_new), _t(batch.slot_mapping), kc, vc,
                                ks, vs, err_word=err)
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
    saved = os.environ.pop("PKV_PREFIX_PASS", None)
    if pass_ is not None:
        os.environ["PKV_PREFIX_PASS"] = pass_
    try:
        out = pkv.paged_decode_attention_prefix_shared_fp8(
            _t(batch.q), kc, vc, _t(batch.block_tables), _t(batch.context_lens), batch.scale, ks,
            vs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size, _t(offs),
            _t(pref), gmax, pmax, max_context_len=batch.max_context_len, lse=lse, err_word=err)
    finally:
        os.environ.pop("PKV_PREFIX_PASS", None)
        if saved is not None:
            os.environ["PKV_PREFIX_PASS"] = saved
    bits = pkv.get_error(err)
    return out.cpu().numpy(), lse.cpu().numpy().astype(np.float64), bits


@pytest.mark.parametrize("pass_", ["shared", None])
@pytest.mark.parametrize("cfg", [3, 5])
def test_fp8_prefix_shared_workloads(cfg, pass_):
    """Full-size shared-prefix workloads with E4M3 caches, poisoned: every
    output and lse of the prefix-aware call against the oracle's E4M3 decode,
    through the two-pass path and the library's choice."""
    batch = wl.workload(cfg, poison=True)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    out, lse, bits = gpu_f8_shared(batch, kc8, vc8, ks, vs, pass_=pass_)
    assert bits == 0
    ref = oracle_f8(batch, kc8, vc8, ks, vs)
    assert_close(out, ref["out"], what=f"fp8 prefix-aware workload {cfg}")
    assert np.max(np.abs(lse - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_fp8_prefix_shared_edge_cases(d, g):
    """Groups of 5 (one member shorter than the prefix), 2 (no private tile:
    the output is the shared pass's alone, its columns mapped back from the
    E4M3 tile math's order), 1, and 3 with a prefix that is no whole tile."""
    rng = np.random.default_rng(900 + 10 * d + g)
    Hk = 2
    lens = [100, 60, 33, 130, 75, 64, 64, 40, 90, 91, 70]
    shared = [([0, 1, 2, 3, 4], 3), ([5, 6], 4), ([8, 9, 10], 3)]
    batch = wl.make_batch("f8edge", lens, Hk * g, Hk, d, 16, rng, append=False, poison=True,
                          shared=shared)
    groups = (np.array([0, 5, 7, 8, 11], dtype=np.int32), np.array([48, 64, 0, 37], dtype=np.int32),
              5, 64)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    out, lse, bits = gpu_f8_shared(batch, kc8, vc8, ks, vs, groups)
    assert bits == 0
    ref = oracle_f8(batch, kc8, vc8, ks, vs)
    assert_close(out, ref["out"], what=f"fp8 prefix-aware d={d} g={g}")
    assert np.max(np.abs(lse - ref["lse"])) <= 1e-4
    # the regular E4M3 call on the same caches agrees
    reg = gpu_f8(batch, kc8, vc8, ks, vs)
    assert np.max(np.abs(out.astype(np.float64) - reg["out"].astype(np.float64))) <= 2e-3


@pytest.mark.parametrize("cfg", [2, 5])
def test_fp8_tables_ready_flag(cfg):
    """paged_decode_attention_fp8_ex and the prefix-aware E4M3 call with
    PKV_TABLES_READY, back to back: bit-identical to the calls without it."""
    batch = wl.workload(cfg, poison=True)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    kc, vc = _t(kc8), _t(vc8)
    q, bt, cl = _t(batch.q), _t(batch.block_tables), _t(batch.context_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if batch.has_append:  # the kernel just before the first call writes the caches
        pkv.paged_kv_append_fp8(_t(batch.k_new), _t(batch.v_new), _t(batch.slot_mapping), kc, vc,
                                ks, vs, err_word=err)
    outs = []
    for flags in (pkv.PKV_TABLES_READY, pkv.PKV_TABLES_READY, 0):
        outs.append(pkv.paged_decode_attention_fp8(
            q, kc, vc, bt, cl, batch.scale, ks, vs, batch.n_q_heads, batch.n_kv_heads,
            batch.head_dim, batch.block_size, max_context_len=batch.max_context_len,
            err_word=err, flags=flags).cpu().numpy())
    if batch.meta.get("shared"):
        offs, pref, gmax, pmax = wl.prefix_groups(batch)
        for flags in (pkv.PKV_TABLES_READY, 0):
            outs.append(pkv.paged_decode_attention_prefix_shared_fp8(
                q, kc, vc, bt, cl, batch.scale, ks, vs, batch.n_q_heads, batch.n_kv_heads,
                batch.head_dim, batch.block_size, _t(offs), _t(pref), gmax, pmax,
                max_context_len=batch.max_context_len, err_word=err, flags=flags).cpu().numpy())
        assert np.array_equal(outs[3].view(np.uint16), outs[4].view(np.uint16))
    assert pkv.get_error(err) == 0
    for o in outs[1:3]:
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16))
    ref = oracle_f8(batch, kc8, vc8, ks, vs)
    assert_close(outs[0], ref["out"], what=f"flagged fp8 workload {cfg}")


def _step8(batch, kc8, vc8, ks, vs, flags, slot_mapping=None, context_lens=None):
    """paged_decode_step_fp8 on fresh device copies: out, lse, caches, bits."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
    kc, vc = _t(kc8), _t(vc8)
    sm = _t(batch.slot_mapping if slot_mapping is None else slot_mapping)
    cl = _t(batch.context_lens if context_lens is None else context_lens)
    out = pkv.paged_decode_step_fp8(
        _t(batch.k_new), _t(batch.v_new), sm, _t(batch.q), kc, vc, _t(batch.block_tables), cl,
        batch.scale, ks, vs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
        batch.block_size, max_context_len=batch.max_context_len, lse=lse, err_word=err,
        flags=flags)
    bits = pkv.get_error(err)
    return out.cpu().numpy(), lse.cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy(), bits


STEP_FLAGS = (pkv.PKV_APPEND_NEWEST, pkv.PKV_APPEND_NEWEST | pkv.PKV_TABLES_READY)


def _same8(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8),
                          np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("cfg", [1, 2])
def test_fp8_step_matches_separate_calls(cfg):
    """paged_decode_step_fp8 (the append kernel, then the attention with its
    prologue under the append): codes, output and lse bit-identical to the
    separate calls, with and without the step flags."""
    batch = wl.workload(cfg, poison=True)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    two = _step8(batch, kc8, vc8, ks, vs, 0)
    assert two[4] == 0
    sep = gpu_f8(batch, kc8, vc8, ks, vs)
    assert _same8(two[0], sep["out"]) and _same8(two[2], sep["k_cache"])
    assert _same8(two[3], sep["v_cache"])
    for flags in STEP_FLAGS:
        got = _step8(batch, kc8, vc8, ks, vs, flags)
        assert got[4] == 0, flags
        for x, y in zip(got[:4], two[:4]):
            assert _same8(x, y), flags
    ref = oracle_f8(batch, kc8, vc8, ks, vs)
    assert_close(two[0], ref["out"], what=f"fp8 step workload {cfg}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32, 64])
def test_fp8_step_edge_shapes(d, g, bs):
    rng = np.random.default_rng(700 + d + 10 * g + bs)
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 64, 130, 300, 1000]
    batch = wl.make_batch("f8step", lens, 2 * g, 2, d, bs, rng, append=True, poison=True)
    ks, vs = _scales(batch)
    kc8, vc8 = _caches8(batch, ks, vs)
    two = _step8(batch, kc8, vc8, ks, vs, 0)
    assert two[4] == 0
    for flags in STEP_FLAGS:
        got = _step8(batch, kc8, vc8, ks, vs, flags)
        assert got[4] == 0
        for x, y in zip(got[:4], two[:4]):
            assert _same8(x, y), (d, g, bs, flags)
    assert_close(two[0], oracle_f8(batch, kc8, vc8, ks, vs)["out"],
                 what=f"fp8 step d={d} g={g} bs={bs}")
