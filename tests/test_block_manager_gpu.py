"""Parallel sampling end to end on the GPU: prompts prefilled through the
block manager, forked into completions that share the prompt blocks
(reference count 4), one decode step with copy-on-write of the shared tail
(paged_kv_copy_blocks), the append and the attention, then a second step.
The cache is compared bit for bit with a CPU replay of the same copies and
writes, and the attention with the oracle and with dense attention over the
logical sequences."""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_213_gb300 as pkv
from gpu_util import assert_close
from paged_kv_cache_213_gb300.blocks import BlockManager, paged_kv_copy_blocks
from pins import dense_reference

pytestmark = pytest.mark.gpu


def test_fork_cow_decode_matches_dense():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(42)
    NB, bs, H, Hk, d = 96, 16, 16, 2, 128
    scale = 1.0 / np.sqrt(d)
    prompts = [50, 33]
    kids = 3
    bm = BlockManager(NB, bs)
    kc = torch.zeros(NB, Hk, bs, d, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    kc_cpu = np.zeros((NB, Hk, bs, d), dtype=np.float16)
    vc_cpu = np.zeros_like(kc_cpu)
    logical_k, logical_v, seqs = {}, {}, []

    def write(tokens):
        """tokens: list of (seq, slot, copy, k_row, v_row); copies first."""
        copies = [t[2] for t in tokens if t[2] is not None]
        if copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device="cuda")
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device="cuda")
            rows = torch.tensor([c[2] for c in copies], dtype=torch.int32, device="cuda")
            paged_kv_copy_blocks(kc, vc, src, dst, rows)
            for s_, d_, n_ in copies:
                kc_cpu[d_, :, :n_] = kc_cpu[s_, :, :n_]
                vc_cpu[d_, :, :n_] = vc_cpu[s_, :, :n_]
        kn = np.stack([t[3] for t in tokens])
        vn = np.stack([t[4] for t in tokens])
        slots = np.array([t[1] for t in tokens], dtype=np.int64)
        pkv.paged_kv_append(torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(),
                            torch.from_numpy(slots).cuda(), kc, vc)
        k2, v2 = oracle.append(kn, vn, slots, kc_cpu, vc_cpu, bs)
        kc_cpu[:] = k2
        vc_cpu[:] = v2

    # prefill the prompts
    for p, L in enumerate(prompts):
        sid = 100 * p
        bm.add_sequence(sid)
        seqs.append(sid)
        toks = []
        ks = rng.standard_normal((L, Hk, d)).astype(np.float16)
        vs = rng.standard_normal((L, Hk, d)).astype(np.float16)
        for t in range(L):
            slot, copy = bm.append_slot(sid)
            assert copy is None
            toks.append((sid, slot, None, ks[t], vs[t]))
        write(toks)
        logical_k[sid], logical_v[sid] = list(ks), list(vs)
        for c in range(1, kids + 1):
            bm.fork(sid, sid + c)
            seqs.append(sid + c)
            logical_k[sid + c] = list(ks)
            logical_v[sid + c] = list(vs)
    prompt_tail = {100 * p: bm.block_table(100 * p)[-1] for p in range(len(prompts))}
    assert all(bm.block_info(b)[0] == kids + 1 for b in prompt_tail.values())

    def step(order):
        toks = []
        for sid in order:
            slot, copy = bm.append_slot(sid)
            k = rng.standard_normal((Hk, d)).astype(np.float16)
            v = rng.standard_normal((Hk, d)).astype(np.float16)
            toks.append((sid, slot, copy, k, v))
            logical_k[sid].append(k)
            logical_v[sid].append(v)
        write(toks)
        return toks

    def attend():
        B = len(seqs)
        lens = np.array([bm.length(s) for s in seqs], dtype=np.int32)
        MB = max(len(bm.block_table(s)) for s in seqs)
        bt = np.full((B, MB), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            t = bm.block_table(s)
            bt[i, :len(t)] = t
        q = rng.standard_normal((B, H, d)).astype(np.float16)
        out = pkv.paged_decode_attention(torch.from_numpy(q).cuda(), kc, vc,
                                         torch.from_numpy(bt).cuda(),
                                         torch.from_numpy(lens).cuda(), scale, H, Hk, d, bs,
                                         max_context_len=int(lens.max()))
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ref, _, _ = oracle.decode(q, kc_cpu, vc_cpu, bt, lens, scale, H, Hk, d, bs)
        assert_close(got, ref, what="vs oracle")
        Lmax = int(lens.max())
        K = np.zeros((B, Hk, Lmax, d), dtype=np.float16)
        V = np.zeros_like(K)
        for i, s in enumerate(seqs):
            K[i, :, :lens[i]] = np.stack(logical_k[s]).transpose(1, 0, 2)
            V[i, :, :lens[i]] = np.stack(logical_v[s]).transpose(1, 0, 2)
        dense, _ = dense_reference(q, K, V, lens, scale, H, Hk)
        assert_close(got, dense, what="vs dense logical attention")

    # decode step 1: children first (copy-on-write), parents last (in place)
    order = [s for s in seqs if s % 100] + [s for s in seqs if s % 100 == 0]
    toks = step(order)
    cows = [t for t in toks if t[2] is not None]
    assert len(cows) == kids * len(prompts)
    assert all(t[2][2] == prompts[t[0] // 100] % bs for t in cows)
    for p in range(len(prompts)):
        assert bm.block_table(100 * p)[-1] == prompt_tail[100 * p]  # parent kept its tail
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), kc_cpu.view(np.uint16))
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), vc_cpu.view(np.uint16))
    attend()
    # decode step 2: every tail is private now, no copies
    toks = step(seqs)
    assert all(t[2] is None for t in toks)
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), kc_cpu.view(np.uint16))
    attend()


def test_prefix_groups_from_manager_drive_prefix_aware_attention():
    """Parallel sampling built through the block manager (prompts prefilled,
    forked into four completions, each decoding its own tokens with
    copy-on-write of the shared tail), then attended through the prefix-aware
    entry point with the groups the manager reports: equal to the oracle and
    to the regular entry point."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(5)
    NB, bs, H, Hk, d = 1024, 16, 64, 8, 128
    scale = 1.0 / np.sqrt(d)
    bm = BlockManager(NB, bs)
    kc = torch.zeros(NB, Hk, bs, d, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)

    def write(slots, copies):
        if copies:
            src = torch.tensor([c[0] for c in copies], dtype=torch.int32, device="cuda")
            dst = torch.tensor([c[1] for c in copies], dtype=torch.int32, device="cuda")
            rows = torch.tensor([c[2] for c in copies], dtype=torch.int32, device="cuda")
            paged_kv_copy_blocks(kc, vc, src, dst, rows)
        n = len(slots)
        kn = torch.from_numpy(rng.standard_normal((n, Hk, d)).astype(np.float16)).cuda()
        vn = torch.from_numpy(rng.standard_normal((n, Hk, d)).astype(np.float16)).cuda()
        pkv.paged_kv_append(kn, vn, torch.tensor(slots, dtype=torch.int64, device="cuda"), kc, vc)

    order = []
    for p, L in enumerate((500, 777, 33, 260)):
        root = 10 * p
        bm.add_sequence(root)
        write([bm.append_slot(root)[0] for _ in range(L)], [])
        fam = [root] + [root + c for c in (1, 2, 3)]
        for c in fam[1:]:
            bm.fork(root, c)
        for _ in range(20):  # each completion decodes its own tokens
            slots, copies = [], []
            for s in fam:
                slot, copy = bm.append_slot(s)
                slots.append(slot)
                if copy is not None:
                    copies.append(copy)
            write(slots, copies)
        order += fam
    offs, pref, gmax, pmax = bm.prefix_groups(order)
    assert list(np.diff(offs)) == [4, 4, 4, 4] and gmax == 4
    assert list(pref) == [496, 768, 32, 256]  # the prompts' full blocks
    lens = np.array([bm.length(s) for s in order], dtype=np.int32)
    MB = max(len(bm.block_table(s)) for s in order)
    bt = np.full((len(order), MB), -1, dtype=np.int32)
    for i, s in enumerate(order):
        t = bm.block_table(s)
        bt[i, :len(t)] = t
    q = rng.standard_normal((len(order), H, d)).astype(np.float16)
    dq, dbt, dcl = (torch.from_numpy(x).cuda() for x in (q, bt, lens))
    # the two-pass path (these prefixes are small enough that the library
    # would otherwise pick the regular attention, whose L2 hits share them)
    os.environ["PKV_PREFIX_PASS"] = "shared"
    try:
        shared = pkv.paged_decode_attention_prefix_shared(
            dq, kc, vc, dbt, dcl, scale, H, Hk, d, bs, torch.from_numpy(offs).cuda(),
            torch.from_numpy(pref).cuda(), gmax, pmax, max_context_len=int(lens.max()))
    finally:
        del os.environ["PKV_PREFIX_PASS"]
    regular = pkv.paged_decode_attention(dq, kc, vc, dbt, dcl, scale, H, Hk, d, bs,
                                         max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    ref, _, _ = oracle.decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, scale, H, Hk, d,
                              bs)
    assert_close(shared.cpu().numpy(), ref, what="prefix-aware, manager groups")
    assert_close(regular.cpu().numpy(), ref, what="regular")
