"""Parity of the CUDA paged decode attention (through the C ABI) with the CPU
oracle: the five standard workloads at full size, forced split-K partition
sizes, edge shapes, NaN-poisoned unused memory, bit-exact cases, invariances
and device-flagged index errors."""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_213_gb300 as pkv
from gpu_util import assert_close, compare, gpu_step, oracle_step, relayout, to_dev
from paged_kv_cache_213_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.library()


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_parity(cfg):
    """Full-size workloads, poisoned, in the automatic launch configuration
    the benchmark uses; every output and every lse of the batch compared."""
    batch = wl.workload(cfg, poison=True)
    g = gpu_step(batch)
    assert g["err"] == 0
    ref = oracle_step(batch)
    assert_close(g["out"], ref["out"], what=f"workload {cfg}")
    assert np.max(np.abs(g["lse"] - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("cfg", [1, 2])
def test_append_bitexact_whole_pool(cfg):
    batch = wl.workload(cfg, poison=True)
    g = gpu_step(batch)
    ref = oracle_step(batch, mask=np.zeros((batch.num_seqs, batch.n_q_heads), dtype=bool))
    kc = g["dev"]["k_cache"].cpu().numpy().view(np.uint16)
    vc = g["dev"]["v_cache"].cpu().numpy().view(np.uint16)
    assert np.array_equal(kc, ref["k_cache"].view(np.uint16))
    assert np.array_equal(vc, ref["v_cache"].view(np.uint16))


def test_append_padding_and_bad_slot():
    rng = np.random.default_rng(7)
    batch = wl.make_batch("pad", [5, 16, 17, 33], 8, 2, 128, 16, rng, append=True, poison=True,
                          append_padding=5)
    dev = to_dev(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                        dev["v_cache"], err_word=err)
    assert pkv.get_error(err) == 0
    ref = oracle_step(batch, mask=np.zeros((4, 8), dtype=bool))
    assert np.array_equal(dev["k_cache"].cpu().numpy().view(np.uint16),
                          ref["k_cache"].view(np.uint16))
    assert np.array_equal(dev["v_cache"].cpu().numpy().view(np.uint16),
                          ref["v_cache"].view(np.uint16))
    # a slot beyond the pool is flagged and skipped; everything else lands
    before = dev["k_cache"].clone()
    slots = dev["slot_mapping"].clone()
    slots[0] = batch.num_blocks * batch.block_size + 3
    pkv.paged_kv_append(dev["k_new"], dev["v_new"], slots, dev["k_cache"], dev["v_cache"],
                        err_word=err)
    assert pkv.get_error(err) & pkv.PKV_ERRBIT_SLOT
    assert torch.equal(before.view(torch.int16), dev["k_cache"].view(torch.int16))


@pytest.mark.parametrize("P", [16, 32, 64, 128, 512, 0])
def test_forced_partitions(P):
    """Split-K partition sizes from one tile per partition to one partition
    per sequence: the LSE merge path and the direct path agree with the oracle."""
    rng = np.random.default_rng(100 + P)
    lens = [1, 15, 16, 17, 100, 255, 256, 257, 700]
    batch = wl.make_batch("split", lens, 16, 4, 128, 16, rng, append=True, poison=True)
    g = gpu_step(batch, partition_tokens=P)
    assert g["err"] == 0
    ref = oracle_step(batch)
    assert_close(g["out"], ref["out"], what=f"P={P}")
    assert np.max(np.abs(g["lse"] - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [1, 2, 8, 16, 32])
def test_edge_shapes(d, g, bs):
    rng = np.random.default_rng(1000 * d + 10 * g + bs)
    Hk = 2
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 130]
    batch = wl.make_batch("edge", lens, Hk * g, Hk, d, bs, rng, append=True, poison=True)
    for P in (0, max(16, bs)):
        out = gpu_step(batch, partition_tokens=P)
        assert out["err"] == 0
        ref = oracle_step(batch)
        assert_close(out["out"], ref["out"], what=f"d={d} g={g} bs={bs} P={P}")


def test_empty_sequences():
    rng = np.random.default_rng(3)
    batch = wl.make_batch("empty", [0, 5, 0, 40], 8, 2, 128, 16, rng, append=False, poison=True,
                          max_blocks_per_seq=4)
    for P in (0, 16):
        g = gpu_step(batch, partition_tokens=P)
        assert g["err"] == 0
        assert np.all(g["out"][[0, 2]] == 0)
        assert np.all(np.isneginf(g["lse"][[0, 2]]))
        ref = oracle_step(batch)
        assert_close(g["out"], ref["out"], what="empty")


def test_single_token_is_bitexact():
    """L = 1: the softmax weight is exactly 1, so out == V_0 bit for bit."""
    rng = np.random.default_rng(4)
    batch = wl.make_batch("one", [1] * 12, 32, 8, 128, 16, rng, append=True, poison=True)
    g = gpu_step(batch)
    ref = oracle_step(batch)
    assert np.array_equal(g["out"].view(np.uint16), ref["out16"].view(np.uint16))
    # and the value is the appended V row
    vn = batch.v_new.astype(np.float16)
    for b in range(12):
        for h in range(32):
            assert np.array_equal(g["out"][b, h].view(np.uint16), vn[b, h // 4].view(np.uint16))


def test_dominant_logit_gathers_exact_row():
    """A huge scale makes the softmax one-hot on the arg-max token: the output
    is that token's V row bit for bit -- the gather through the block table
    picks exactly the oracle's row, across partitions."""
    rng = np.random.default_rng(5)
    lens = [40, 300, 1000, 77]
    batch = wl.make_batch("onehot", lens, 8, 2, 128, 16, rng, scale=4000.0, append=True,
                          poison=True)
    ref = oracle_step(batch)
    # logits in double from the appended cache, to find clear winners
    kc = ref["k_cache"].astype(np.float64)
    checked = 0
    for P in (0, 64):
        g = gpu_step(batch, partition_tokens=P)
        assert g["err"] == 0
        for b, L in enumerate(lens):
            t = np.arange(L)
            rows = kc[batch.block_tables[b, t // 16], :, t % 16, :]  # [L, Hk, d]
            for h in range(8):
                s = rows[:, h // 4, :] @ batch.q[b, h].astype(np.float64)
                top2 = np.sort(s)[-2:]
                if top2[1] - top2[0] < 0.05:
                    continue
                assert np.array_equal(g["out"][b, h].view(np.uint16),
                                      ref["out16"][b, h].view(np.uint16))
                checked += 1
    assert checked > 20


def test_invariances_are_bitwise():
    """Physical block order, block size 16 vs 32 and shared vs copied prefix
    blocks do not change a single output bit (a kernel sums in logical order
    whatever the addresses).  Block sizes 1 and 8 run the CUDA-core kernel, so
    they are held to the tolerance here and to bit equality in
    test_kernel_variants_gpu.py, where both sides run that kernel."""
    rng = np.random.default_rng(6)
    lens = [70, 16, 530, 33]
    base = wl.make_batch("inv", lens, 16, 4, 128, 16, rng, append=False, poison=True)
    out0 = gpu_step(base, partition_tokens=64)["out"]
    ref = oracle_step(base)["out"]
    for bs, seed in ((16, 60), (32, 61)):
        out = gpu_step(relayout(base, bs, seed), partition_tokens=64)["out"]
        assert np.array_equal(out.view(np.uint16), out0.view(np.uint16)), f"bs={bs}"
    for bs, seed in ((1, 62), (8, 63)):
        out = gpu_step(relayout(base, bs, seed), partition_tokens=64)["out"]
        assert_close(out, ref, what=f"bs={bs}")
    # shared prefix: make the first 32 tokens of sequences 0 and 2 identical
    base.k_cache[base.block_tables[2, :2]] = base.k_cache[base.block_tables[0, :2]]
    base.v_cache[base.block_tables[2, :2]] = base.v_cache[base.block_tables[0, :2]]
    copied = gpu_step(base, partition_tokens=64)["out"]
    shared = relayout(base, 16, 64, shared=[([0, 2], 2)])
    assert shared.block_tables[0, 0] == shared.block_tables[2, 0]
    out = gpu_step(shared, partition_tokens=64)["out"]
    assert np.array_equal(out.view(np.uint16), copied.view(np.uint16))


def test_bad_block_id_and_length_are_flagged():
    rng = np.random.default_rng(8)
    batch = wl.make_batch("bad", [40, 20], 8, 2, 128, 16, rng, append=False, poison=False)
    batch.block_tables[0, 1] = batch.num_blocks + 5
    g = gpu_step(batch)
    assert g["err"] & pkv.PKV_ERRBIT_BLOCK_ID
    ok = oracle_step(batch, mask=np.array([[False] * 8, [True] * 8]))
    assert_close(g["out"][1], ok["out"][1], what="untouched sequence")
    batch = wl.make_batch("bad", [40, 20], 8, 2, 128, 16, rng, append=False, poison=False)
    batch.context_lens[1] = batch.max_blocks_per_seq * 16 + 1
    g = gpu_step(batch, max_context_len=0)
    assert g["err"] & pkv.PKV_ERRBIT_CONTEXT


def test_host_side_errors():
    rng = np.random.default_rng(9)
    batch = wl.make_batch("h", [300], 8, 2, 128, 16, rng, append=False, poison=False)
    dev = to_dev(batch)
    P, ws = pkv.decode_plan(1, 8, 2, 128, 16, batch.max_blocks_per_seq, 300, 64)
    assert P == 64 and ws > 0
    small = torch.empty(ws - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["context_lens"], 0.1, 8, 2, 128, 16, max_context_len=300,
                                   partition_tokens=64, workspace=small)
    assert e.value.status == -3
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["context_lens"], 0.1, 8, 2, 128, 16, partition_tokens=24)


def test_side_stream_and_reuse():
    """Works on a non-default stream and with a caller-owned workspace reused
    across calls."""
    batch = wl.workload(1, poison=True)
    ref = oracle_step(batch)
    dev = to_dev(batch)
    s = torch.cuda.Stream()
    P, ws = pkv.decode_plan(batch.num_seqs, 4, 2, 64, 16, batch.max_blocks_per_seq,
                            batch.max_context_len, 16)
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"])
        outs = [pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                           dev["block_tables"], dev["context_lens"], batch.scale,
                                           4, 2, 64, 16, max_context_len=batch.max_context_len,
                                           partition_tokens=16, workspace=work)
                for _ in range(3)]
    s.synchronize()
    for o in outs:
        assert_close(o.cpu().numpy(), ref["out"], what="side stream")
    assert np.array_equal(outs[0].cpu().numpy().view(np.uint16),
                          outs[2].cpu().numpy().view(np.uint16))
    assert math.isfinite(float(compare(outs[1].cpu().numpy(), ref["out"])[0]))


@pytest.mark.parametrize("lens_kind", ["many_short", "single_unit", "mixed_empty", "over_2048"])
def test_balanced_split_shapes(lens_kind):
    """The default (balanced) split with segments much shorter than a warp's
    range, a single unit of work, empty sequences mixed in, and a batch too
    large for the balanced kernel (falls back to the partition grid)."""
    rng = np.random.default_rng({"many_short": 1, "single_unit": 2, "mixed_empty": 3,
                                 "over_2048": 4}[lens_kind])
    if lens_kind == "many_short":
        lens = rng.integers(1, 41, size=700)
        H, Hk, d = 8, 2, 128
    elif lens_kind == "single_unit":
        lens = [1]
        H, Hk, d = 4, 1, 64
    elif lens_kind == "mixed_empty":
        lens = [0, 3000, 0, 0, 17, 1, 0, 900, 0]
        H, Hk, d = 32, 8, 128
    else:
        lens = rng.integers(1, 70, size=2100)
        H, Hk, d = 4, 1, 64
    batch = wl.make_batch(lens_kind, lens, H, Hk, d, 16, rng, append=False, poison=True)
    g = gpu_step(batch)
    assert g["err"] == 0
    ref = oracle_step(batch)
    assert_close(g["out"], ref["out"], what=lens_kind)
    fin = np.isfinite(ref["lse"])
    assert np.max(np.abs(g["lse"][fin] - ref["lse"][fin])) <= 1e-4
    assert np.all(np.isneginf(g["lse"][~fin]))


def test_balanced_workspace_reuse_across_plans():
    """One zero-filled workspace serves calls with different shapes in a row:
    the per-segment arrival counters are left at zero by every call."""
    batches = [wl.workload(2, poison=True), wl.workload(3, poison=True),
               wl.make_batch("r", [5000, 17, 3000], 32, 8, 128, 16,
                             np.random.default_rng(9), append=False, poison=True)]
    sizes = []
    for bt in batches:
        P, ws = pkv.decode_plan(bt.num_seqs, bt.n_q_heads, bt.n_kv_heads, bt.head_dim,
                                bt.block_size, bt.max_blocks_per_seq, bt.max_context_len, 0)
        assert P == 0
        sizes.append(ws)
    work = torch.zeros(max(sizes), dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for bt in batches:
            dev = to_dev(bt)
            if bt.has_append:
                pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"],
                                    dev["k_cache"], dev["v_cache"])
            out = pkv.paged_decode_attention(
                dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                dev["context_lens"], bt.scale, bt.n_q_heads, bt.n_kv_heads, bt.head_dim,
                bt.block_size, max_context_len=bt.max_context_len, workspace=work)
            ref = oracle_step(bt)
            assert_close(out.cpu().numpy(), ref["out"], what=f"{bt.name} rep {rep}")
    counters = work[: 16384 * 4].view(torch.int32)
    assert int(counters.abs().sum()) == 0


@pytest.mark.parametrize("cfg", [1, 2])
def test_decode_step_matches_append_then_attend(cfg):
    """paged_decode_step (append, then attention whose prologue overlaps it)
    gives the caches and outputs of the two calls, and matches the oracle."""
    batch = wl.workload(cfg, poison=True)
    dev = to_dev(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.zeros(batch.num_seqs, batch.n_q_heads, device="cuda")
    out = pkv.paged_decode_step(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["q"],
                                dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                dev["context_lens"], batch.scale, batch.n_q_heads,
                                batch.n_kv_heads, batch.head_dim, batch.block_size,
                                max_context_len=batch.max_context_len, lse=lse, err_word=err)
    assert pkv.get_error(err) == 0
    two = gpu_step(batch)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), two["out"].view(np.uint16))
    assert np.array_equal(dev["k_cache"].cpu().numpy().view(np.uint16),
                          two["dev"]["k_cache"].cpu().numpy().view(np.uint16))
    ref = oracle_step(batch)
    assert_close(out.cpu().numpy(), ref["out"], what=f"step {cfg}")
    assert np.max(np.abs(lse.cpu().numpy() - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_tables_ready_flag(cfg):
    """paged_decode_attention_ex with PKV_TABLES_READY, launched right after
    kernels that write the caches (the append) or the workspace (its zero
    fill), then back to back with itself on one workspace: bit-identical to
    the plain call, and the oracle's result, every output."""
    batch = wl.workload(cfg, poison=True)
    dev = to_dev(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, ws = pkv.decode_plan(batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                            batch.block_size, batch.max_blocks_per_seq, batch.max_context_len, 0)
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    work.zero_()  # the kernel just before the first call writes the workspace
    if batch.has_append:  # ... or the caches
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"], err_word=err)

    def call(flags):
        lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
        out = pkv.paged_decode_attention(
            dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
            batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
            max_context_len=batch.max_context_len, workspace=work, lse=lse, err_word=err,
            flags=flags)
        return out, lse
    first = call(pkv.PKV_TABLES_READY)
    second = call(pkv.PKV_TABLES_READY)
    plain = call(0)
    assert pkv.get_error(err) == 0
    o1, l1 = (t.cpu().numpy() for t in first)
    for o, l in (second, plain):
        assert np.array_equal(o.cpu().numpy().view(np.uint16), o1.view(np.uint16))
        assert np.array_equal(l.cpu().numpy(), l1)
    ref = oracle_step(batch)
    assert_close(o1, ref["out"], what=f"flagged workload {cfg}")
    assert np.max(np.abs(l1.astype(np.float64) - ref["lse"])) <= 1e-4


@pytest.mark.parametrize("what", ["tables", "lengths", "both"])
def test_plain_call_after_a_kernel_that_rewrites_the_tables(what):
    """A plain call plans its split before its dependency wait and checks the
    lengths and block ids it read once the wait is over; when the kernel just
    before it rewrites them (here an elementwise kernel storing the real
    values over stale ones), the call must attend over the new ones."""
    batch = wl.workload(2, poison=True)
    dev = to_dev(batch)
    pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                        dev["v_cache"])
    good_bt, good_cl = dev["block_tables"].clone(), dev["context_lens"].clone()
    stale_bt = good_bt.flip(0).contiguous()  # other sequences' (valid) block ids
    stale_cl = (good_cl // 2 + 1).contiguous()
    ref = oracle_step(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, ws = pkv.decode_plan(batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                            batch.block_size, batch.max_blocks_per_seq, batch.max_context_len, 0)
    work = torch.zeros(ws, dtype=torch.uint8, device="cuda")
    for _ in range(4):
        if what in ("tables", "both"):
            dev["block_tables"].copy_(stale_bt)
        if what in ("lengths", "both"):
            dev["context_lens"].copy_(stale_cl)
        torch.cuda.synchronize()
        # the kernels just before the call write the real values
        if what in ("tables", "both"):
            torch.add(good_bt, 0, out=dev["block_tables"])
        if what in ("lengths", "both"):
            torch.add(good_cl, 0, out=dev["context_lens"])
        out = pkv.paged_decode_attention(
            dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
            batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
            max_context_len=batch.max_context_len, workspace=work, err_word=err)
        assert pkv.get_error(err) == 0
        assert_close(out.cpu().numpy(), ref["out"], what=f"after rewritten {what}")


def _run_step(batch, flags, slot_mapping=None, context_lens=None):
    """paged_decode_step on fresh device copies; numpy out, lse, caches, bits."""
    dev = to_dev(batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse = torch.full((batch.num_seqs, batch.n_q_heads), float("nan"), device="cuda")
    sm = dev["slot_mapping"] if slot_mapping is None else torch.from_numpy(slot_mapping).cuda()
    cl = dev["context_lens"] if context_lens is None else torch.from_numpy(context_lens).cuda()
    out = pkv.paged_decode_step(dev["k_new"], dev["v_new"], sm, dev["q"], dev["k_cache"],
                                dev["v_cache"], dev["block_tables"], cl, batch.scale,
                                batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                                batch.block_size, max_context_len=batch.max_context_len,
                                lse=lse, err_word=err, flags=flags)
    bits = pkv.get_error(err)
    return (out.cpu().numpy(), lse.cpu().numpy(), dev["k_cache"].cpu().numpy(),
            dev["v_cache"].cpu().numpy(), bits)


def _same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8),
                          np.ascontiguousarray(b).view(np.uint8))


FUSED = (pkv.PKV_APPEND_NEWEST, pkv.PKV_APPEND_NEWEST | pkv.PKV_TABLES_READY)


@pytest.mark.parametrize("cfg", [1, 2])
def test_fused_append_step_matches_two_kernel_step(cfg):
    """PKV_APPEND_NEWEST: the attention kernel appends each sequence's newest
    token itself (one launch).  Output, lse and the whole pool are bit-identical
    to the two-kernel step, and the output matches the oracle."""
    batch = wl.workload(cfg, poison=True)
    ref = _run_step(batch, 0)
    assert ref[4] == 0
    for flags in FUSED:
        got = _run_step(batch, flags)
        assert got[4] == 0, flags
        for x, y in zip(got[:4], ref[:4]):
            assert _same_bits(x, y), flags
    assert_close(ref[0], oracle_step(batch)["out"], what=f"workload {cfg} step")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [16, 32, 64])
def test_fused_append_step_edge_shapes(d, g, bs):
    rng = np.random.default_rng(600 + d + 10 * g + bs)
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 64, 130, 300, 1000]
    batch = wl.make_batch("fused", lens, 2 * g, 2, d, bs, rng, append=True, poison=True)
    ref = _run_step(batch, 0)
    assert ref[4] == 0
    for flags in FUSED:
        got = _run_step(batch, flags)
        assert got[4] == 0
        for x, y in zip(got[:4], ref[:4]):
            assert _same_bits(x, y), (d, g, bs, flags)
    assert_close(ref[0], oracle_step(batch)["out"], what=f"fused d={d} g={g} bs={bs}")


def test_fused_append_padding_and_broken_promises():
    rng = np.random.default_rng(611)
    batch = wl.make_batch("fused-edge", [5, 40, 17, 100, 33], 8, 2, 128, 16, rng, append=True,
                          poison=True, pool_extra=0.5)
    used = set(batch.block_tables[b, i] for b in range(batch.num_seqs)
               for i in range((int(batch.context_lens[b]) + 15) // 16))
    free = next(i for i in range(batch.num_blocks) if i not in used)
    sm = batch.slot_mapping.copy()
    sm[1] = -1                  # no token for sequence 1
    sm[2] = free * 16 + 3       # a token away from sequence 2's newest position
    ref = _run_step(batch, 0, slot_mapping=sm)
    assert ref[4] == 0
    for flags in FUSED:
        got = _run_step(batch, flags, slot_mapping=sm)
        assert got[4] == pkv.PKV_ERRBIT_APPEND, got[4]   # only the broken promise
        for x, y in zip(got[:4], ref[:4]):                # the token is still written
            assert _same_bits(x, y), flags
    # a token for an empty sequence is flagged and not written
    cl = batch.context_lens.copy()
    cl[3] = 0
    got = _run_step(batch, pkv.PKV_APPEND_NEWEST, context_lens=cl)
    assert got[4] == pkv.PKV_ERRBIT_APPEND
    assert np.all(got[0][3] == 0) and np.all(np.isneginf(got[1][3]))


def test_tables_ready_reads_q_after_the_wait():
    """Under PKV_TABLES_READY the kernel before may write q: here q is the
    output of the attention call just before (which lets its dependent launch
    early), and the flagged call must read it only after that call is done."""
    batch = wl.workload(2, poison=True)
    dev = to_dev(batch)
    pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                        dev["v_cache"])
    args = (dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
            batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size)
    mcl = batch.max_context_len
    results = []
    for flags in (0, pkv.PKV_TABLES_READY, pkv.PKV_TABLES_READY):
        first = pkv.paged_decode_attention(dev["q"], *args, max_context_len=mcl)
        second = pkv.paged_decode_attention(first, *args, max_context_len=mcl, flags=flags)
        results.append(second.cpu().numpy())
    for r in results[1:]:
        assert np.array_equal(r.view(np.uint16), results[0].view(np.uint16))


def test_pinned_host_out():
    """out may be pinned host memory: the kernels store the results into it
    directly.  The step (one launch and two kernels) and the attention call
    give the same bits as with device memory."""
    batch = wl.workload(2, poison=True)
    shape = (batch.num_seqs, batch.n_q_heads, batch.head_dim)
    outs = []
    for where in ("device", "host"):
        for flags in (0, pkv.PKV_APPEND_NEWEST):
            dev = to_dev(batch)
            out = torch.empty(shape, dtype=torch.float16, pin_memory=True) if where == "host" \
                else None
            got = pkv.paged_decode_step(dev["k_new"], dev["v_new"], dev["slot_mapping"],
                                        dev["q"], dev["k_cache"], dev["v_cache"],
                                        dev["block_tables"], dev["context_lens"], batch.scale,
                                        batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                                        batch.block_size, max_context_len=batch.max_context_len,
                                        out=out, flags=flags)
            att_out = torch.empty(shape, dtype=torch.float16, pin_memory=True) \
                if where == "host" else None
            att = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                             dev["block_tables"], dev["context_lens"],
                                             batch.scale, batch.n_q_heads, batch.n_kv_heads,
                                             batch.head_dim, batch.block_size,
                                             max_context_len=batch.max_context_len, out=att_out)
            torch.cuda.synchronize()
            outs.append((got.cpu().numpy().copy(), att.cpu().numpy().copy()))
    for step_out, att_out in outs[1:]:
        assert np.array_equal(step_out.view(np.uint16), outs[0][0].view(np.uint16))
        assert np.array_equal(att_out.view(np.uint16), outs[0][1].view(np.uint16))
    assert_close(outs[0][0], oracle_step(batch)["out"], what="pinned host out")


def test_copy_in_from_pinned_and_device_memory():
    """paged_copy_in moves bytes into device memory with a kernel, from pinned
    host memory or from device memory, bit for bit."""
    rng = np.random.default_rng(5)
    for n in (16, 4096, 409600, 1 << 22):
        host = torch.from_numpy(rng.integers(0, 256, n, dtype=np.uint8)).pin_memory()
        dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
        pkv.paged_copy_in(dst, host)
        torch.cuda.synchronize()
        assert torch.equal(dst.cpu(), host)
        dst2 = torch.zeros(n, dtype=torch.uint8, device="cuda")
        pkv.paged_copy_in(dst2, dst)
        torch.cuda.synchronize()
        assert torch.equal(dst2, dst)
