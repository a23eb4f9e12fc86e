"""Block manager: the library's C++ manager and the plain-Python oracle
against the serving page's Lab 1 worked example, against each other on
random operation sequences, and against invariants.  Host only (no GPU)."""
import json
import os

import numpy as np
import pytest

from oracle.block_manager import BlockManagerOracle, OutOfBlocks as OracleOOM
from paged_kv_cache_213_gb300 import build as pkv_build

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "cow_lab1.json")))


@pytest.fixture(scope="module")
def cpp():
    pkv_build.build()
    from paged_kv_cache_213_gb300.blocks import BlockManager, OutOfBlocks
    return BlockManager, OutOfBlocks


def _tables(bm, seqs):
    return {s: bm.block_table(s) if hasattr(bm, "block_table") else list(bm.tables[s])
            for s in seqs}


def _info(bm, b):
    if hasattr(bm, "block_info"):
        return bm.block_info(b)
    return bm.ref[b], bm.filled[b]


def run_lab1(bm):
    """Prefill the prompt in the parent, fork three children, decode one token
    in each child and then in the parent.  Returns the facts the page states."""
    g = GOLDEN
    bs = g["block_size"]
    bm.add_sequence(0)
    for _ in range(g["prompt_tokens"]):
        _, copy = bm.append_slot(0)
        assert copy is None
    prompt = list(_tables(bm, [0])[0])
    facts = {"after_prefill": {"table_blocks": len(prompt),
                               "filled": [_info(bm, b)[1] for b in prompt]}}
    for c in (1, 2, 3):
        bm.fork(0, c)
    facts["after_fork"] = {"refcount": [_info(bm, b)[0] for b in prompt]}
    fresh, copies, rows = [], [], []
    for c in (1, 2, 3):
        slot, copy = bm.append_slot(c)
        copies.append(copy)
        tail = _tables(bm, [c])[c][-1]
        fresh.append(tail)
        rows.append(slot - tail * bs)
    slot, copy = bm.append_slot(0)
    last_tail = _tables(bm, [0])[0][-1]
    facts["after_first_decode_step"] = {
        "fresh_blocks": len(set(fresh) - set(prompt)),
        "fresh_block_refcount": sorted({_info(bm, b)[0] for b in fresh})[0],
        "fresh_block_filled": sorted({_info(bm, b)[1] for b in fresh})[0],
        "copied_rows": sorted({cp[2] for cp in copies})[0],
        "divergent_token_row": sorted(set(rows))[0],
        "last_sharer_writes_in_place": copy is None and last_tail == prompt[-1]
                                       and slot == prompt[-1] * bs + 2,
        "shared_tail_filled_after": _info(bm, prompt[-1])[1],
        "shared_tail_refcount_after": _info(bm, prompt[-1])[0],
        "prefix_refcount_after": [_info(bm, b)[0] for b in prompt[:3]],
        "prefix_tokens": sum(_info(bm, b)[1] for b in prompt[:3]),
    }
    # every copy-on-write copied the shared tail into the child's fresh block
    assert all(cp[0] == prompt[-1] and cp[1] == f for cp, f in zip(copies, fresh))
    return facts


def _expected():
    return {k: GOLDEN[k] for k in ("after_prefill", "after_fork", "after_first_decode_step")}


def test_lab1_worked_example_oracle():
    assert run_lab1(BlockManagerOracle(100, 16)) == _expected()


def test_lab1_worked_example_library(cpp):
    BlockManager, _ = cpp
    assert run_lab1(BlockManager(100, 16)) == _expected()


def _random_ops(seed, n_ops=1500, num_blocks=64, bs=4):
    rng = np.random.default_rng(seed)
    ops, live, nxt = [], [], 0
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.08 or not live:
            ops.append(("add", nxt))
            live.append(nxt)
            nxt += 1
        elif r < 0.15:
            p = int(rng.choice(live))
            ops.append(("fork", p, nxt))
            live.append(nxt)
            nxt += 1
        elif r < 0.22:
            s = int(rng.choice(live))
            ops.append(("free", s))
            live.remove(s)
        else:
            ops.append(("append", int(rng.choice(live))))
    return ops, num_blocks, bs


def _apply(bm, op, oom_types):
    try:
        if op[0] == "add":
            bm.add_sequence(op[1])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        elif op[0] == "free":
            bm.free_sequence(op[1])
        else:
            return bm.append_slot(op[1])
    except oom_types:
        return "oom"
    return None


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_library_matches_oracle_on_random_operations(cpp, seed):
    BlockManager, OOM = cpp
    ops, nb, bs = _random_ops(seed)
    a, b = BlockManager(nb, bs), BlockManagerOracle(nb, bs)
    live = set()
    ooms = 0
    for op in ops:
        ra, rb = _apply(a, op, (OOM,)), _apply(b, op, (OracleOOM,))
        assert ra == rb, op
        ooms += ra == "oom"
        if op[0] in ("add", "fork"):
            live.add(op[-1])
        elif op[0] == "free":
            live.discard(op[1])
        assert a.num_free() == b.num_free()
    for s in live:
        assert a.block_table(s) == b.tables[s]
        assert a.length(s) == b.lengths[s]
    for blk in range(nb):
        assert a.block_info(blk) == (b.ref[blk], b.filled[blk])
    assert ooms > 0  # the pool ran dry at least once


@pytest.mark.parametrize("seed", [10, 11])
def test_invariants(seed):
    """Reference counts equal the number of tables holding a block; used +
    free = pool; every sequence's length matches its table and rows."""
    ops, nb, bs = _random_ops(seed, n_ops=1200)
    bm = BlockManagerOracle(nb, bs)
    for op in ops:
        _apply(bm, op, (OracleOOM,))
        holders = {}
        for t in bm.tables.values():
            for blk in t:
                holders[blk] = holders.get(blk, 0) + 1
        assert all(bm.ref[blk] == holders.get(blk, 0) for blk in range(nb))
        assert len(holders) + bm.num_free() == nb
        for s, t in bm.tables.items():
            full = sum(bm.filled[blk] for blk in t[:-1]) + (bm.filled[t[-1]] if t else 0)
            assert full == bm.lengths[s]
            assert all(bm.filled[blk] == bs for blk in t[:-1])


def test_out_of_blocks_leaves_state_unchanged(cpp):
    BlockManager, OOM = cpp
    bm = BlockManager(2, 4)
    bm.add_sequence(7)
    for _ in range(8):
        bm.append_slot(7)
    with pytest.raises(OOM):
        bm.append_slot(7)
    assert bm.length(7) == 8 and bm.num_free() == 0
    bm.fork(7, 8)
    bm.free_sequence(7)
    assert bm.num_free() == 0
    bm.free_sequence(8)
    assert bm.num_free() == 2


def _check_groups(bm, ids, groups):
    """The prefix groups' defining properties, checked on the block tables."""
    offs, pref, most, longest = groups
    tables = [bm.block_table(s) for s in ids]
    bs = bm.block_size
    assert offs[0] == 0 and offs[-1] == len(ids) and np.all(np.diff(offs) >= 1)
    assert len(pref) == len(offs) - 1
    assert most == (int(np.max(np.diff(offs))) if len(ids) else 0)
    assert longest == (int(pref.max()) if len(pref) else 0)
    for gi in range(len(pref)):
        rows = list(range(offs[gi], offs[gi + 1]))
        first = tables[rows[0]]
        nb = int(pref[gi]) // bs
        assert pref[gi] % bs == 0
        if len(rows) == 1:
            assert pref[gi] == 0
            continue
        # every member starts with the first member's first block ...
        assert first and all(tables[r] and tables[r][0] == first[0] for r in rows)
        # ... and holds its first nb blocks, and no longer common run exists
        assert all(tables[r][:nb] == first[:nb] for r in rows)
        assert any(len(tables[r]) <= nb or len(first) <= nb or tables[r][nb] != first[nb]
                   for r in rows[1:])
    # maximal runs: neighbouring groups start with different first blocks
    for gi in range(1, len(pref)):
        a, b = tables[offs[gi] - 1], tables[offs[gi]]
        assert not (a and b and a[0] == b[0])


def test_prefix_groups_properties(cpp):
    BlockManager, _ = cpp
    rng = np.random.default_rng(11)
    for trial in range(40):
        bs = int(rng.choice([1, 4, 16]))
        bm = BlockManager(4096, bs)
        ids, nxt = [], 0
        for _ in range(int(rng.integers(1, 6))):  # prompts, each with forked siblings
            root = nxt
            nxt += 1
            bm.add_sequence(root)
            for _ in range(int(rng.integers(0, 70))):
                bm.append_slot(root)
            fam = [root]
            for _ in range(int(rng.integers(0, 4))):
                child = nxt
                nxt += 1
                bm.fork(int(rng.choice(fam)), child)
                fam.append(child)
            for s in fam:  # diverge by a few tokens each
                for _ in range(int(rng.integers(0, 20))):
                    bm.append_slot(s)
            ids += fam
        if trial % 3 == 0:
            rng.shuffle(ids)  # sharers no longer adjacent: still a valid partition
        _check_groups(bm, ids, bm.prefix_groups(ids))


def test_prefix_groups_of_forked_prompt(cpp):
    """Four completions forked from a 3968-token prompt, two private blocks
    each (the 70B-shaped parallel-sampling batch): one group of four sharing
    the prompt's 248 full blocks."""
    BlockManager, _ = cpp
    bm = BlockManager(2048, 16)
    bm.add_sequence(0)
    for _ in range(3968):
        bm.append_slot(0)
    for c in (1, 2, 3):
        bm.fork(0, c)
    for s in (0, 1, 2, 3):
        for _ in range(32):
            bm.append_slot(s)
    offs, pref, most, longest = bm.prefix_groups([0, 1, 2, 3])
    assert list(offs) == [0, 4] and list(pref) == [3968] and most == 4 and longest == 3968
    offs, pref, _, _ = bm.prefix_groups([0, 1])
    assert list(pref) == [3968]
    with pytest.raises(Exception):
        bm.prefix_groups([0, 77])  # unknown id
