"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes a loaded oracle library (the real one, or a
deliberately broken copy built by the mutation test) and raises
AssertionError (or oracle.OracleError) when the oracle disagrees with:

  * a library routine that computes the same thing by another road
    (torch's float64 scaled_dot_product_attention and scipy's softmax /
    logsumexp on contiguous K/V; numpy's float16 conversions; numpy fancy
    indexing for the scatter of the append);
  * closed forms (one token, zero query, equal keys, two tokens, a dominant
    logit, all-ones values);
  * exact invariances (physical block order, block size 1 vs 16, shared vs
    copied prefix blocks, GQA vs MHA with replicated KV heads);
  * the log-sum-exp merge identity over any split of the token range.

The paged inputs are built here from contiguous logical K/V, so that the
gather the oracle performs is checked against data whose logical order is
known independently.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

import oracle

F16_NAN = np.uint16(0x7E00)


# ----------------------------------------------------------------------------
# input construction from logical (contiguous) K/V
# ----------------------------------------------------------------------------

def randn16(rng, shape):
    return rng.standard_normal(shape).astype(np.float16)


def paginate(K, V, lens, bs, rng, extra_blocks=3, shared=None, poison=True, perm=None):
    """Scatter logical K/V [B, Hk, Lmax, d] into a permuted block pool.

    shared: (members, n_blocks) -- the members' first n_blocks logical blocks
      go to one set of physical blocks (their contents must be equal, the
      caller makes them so).
    Returns k_cache, v_cache [NB, Hk, bs, d] fp16, block_tables [B, MB] int32.
    """
    B, Hk, Lmax, d = K.shape
    nblk = [(int(L) + bs - 1) // bs for L in lens]
    MB = max(1, max(nblk))
    keys = []
    table = [[None] * n for n in nblk]
    if shared is not None:
        members, n_sh = shared
        for lb in range(n_sh):
            key = ("s", lb)
            keys.append((key, members[0], lb))
            for b in members:
                if lb < nblk[b]:
                    table[b][lb] = len(keys) - 1
    for b in range(B):
        for lb in range(nblk[b]):
            if table[b][lb] is None:
                keys.append((("p", b, lb), b, lb))
                table[b][lb] = len(keys) - 1
    NB = len(keys) + extra_blocks
    if perm is None:
        perm = rng.permutation(NB)
    kc = np.zeros((NB, Hk, bs, d), dtype=np.float16)
    vc = np.zeros((NB, Hk, bs, d), dtype=np.float16)
    if poison:
        kc.view(np.uint16)[:] = F16_NAN
        vc.view(np.uint16)[:] = F16_NAN
    for k, (_, b, lb) in enumerate(keys):
        phys = perm[k]
        L = int(lens[b])
        n = min(bs, L - lb * bs)
        kc[phys, :, :n, :] = K[b, :, lb * bs: lb * bs + n, :]
        vc[phys, :, :n, :] = V[b, :, lb * bs: lb * bs + n, :]
    bt = np.full((B, MB), -7 if poison else 0, dtype=np.int32)
    for b in range(B):
        for lb in range(nblk[b]):
            bt[b, lb] = perm[table[b][lb]]
    return kc, vc, bt


def logical_problem(rng, B=3, H=4, Hk=2, d=64, lens=(1, 17, 40), dist="randn"):
    lens = np.asarray(lens)
    Lmax = int(lens.max())
    q = randn16(rng, (B, H, d))
    K = randn16(rng, (B, Hk, Lmax, d))
    V = randn16(rng, (B, Hk, Lmax, d))
    return q, K, V, lens


def dense_reference(q, K, V, lens, scale, H, Hk):
    """Contiguous attention by torch SDPA in float64 and scipy's logsumexp."""
    B, _, d = q.shape
    g = H // Hk
    out = np.zeros((B, H, d))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        qt = torch.from_numpy(q[b].astype(np.float64)).reshape(1, H, 1, d)
        kt = torch.from_numpy(K[b, :, :L].astype(np.float64)).repeat_interleave(g, dim=0)
        vt = torch.from_numpy(V[b, :, :L].astype(np.float64)).repeat_interleave(g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.reshape(1, H, L, d), vt.reshape(1, H, L, d), scale=scale)
        out[b] = o.reshape(H, d).numpy()
        s = np.einsum("hd,hld->hl", q[b].astype(np.float64), kt.numpy()) * scale
        lse[b] = scipy.special.logsumexp(s, axis=1)
    return out, lse


def run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, bs):
    return oracle.decode(q, kc, vc, bt, np.asarray(lens, dtype=np.int32), scale, H, Hk, d, bs,
                         lib=lib)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_fp16_decode(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.pkvo_f16_to_f64(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_fp16_encode(lib, n_random=20000, seed=5):
    rng = np.random.default_rng(seed)
    finite = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = finite.view(np.float16)
    finite = finite[np.isfinite(vals)]
    # exact values round-trip
    for h in finite[:: 7]:
        x = float(np.uint16(h).view(np.float16))
        assert lib.pkvo_f64_to_f16(x) == int(h), hex(int(h))
    # midpoints between neighbours: ties go to the even significand
    pos = np.sort(np.unique(np.abs(vals[np.isfinite(vals)].astype(np.float64))))
    mids = (pos[:-1] + pos[1:]) / 2.0
    xs = np.concatenate([mids[::3], -mids[1::5],
                         rng.standard_normal(n_random) * 10.0 ** rng.integers(-9, 5, n_random),
                         [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                          2.0 ** -24 * 1.5, 2.0 ** -24 * 2.5, -0.0, 0.0]])
    with np.errstate(over="ignore"):  # values from 65520 up round to infinity, as intended
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([lib.pkvo_f64_to_f16(float(x)) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


def pin_dense_sdpa(lib, seed=11):
    """Paged gather + softmax equals contiguous SDPA (float64 library routine)."""
    rng = np.random.default_rng(seed)
    for (B, H, Hk, d, bs, lens) in [(3, 4, 2, 64, 16, (1, 17, 40)),
                                    (2, 8, 1, 128, 16, (33, 16)),
                                    (2, 4, 4, 64, 1, (5, 9)),
                                    (4, 8, 2, 64, 8, (15, 16, 17, 64))]:
        q, K, V, lens = logical_problem(rng, B, H, Hk, d, lens)
        scale = 1.0 / math.sqrt(d)
        kc, vc, bt = paginate(K, V, lens, bs, rng)
        out, lse, out16 = run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, bs)
        ref, ref_lse = dense_reference(q, K, V, lens, scale, H, Hk)
        assert np.max(np.abs(out - ref)) <= 1e-12, np.max(np.abs(out - ref))
        assert np.max(np.abs(lse - ref_lse)) <= 1e-12
        assert np.array_equal(out16.view(np.uint16), ref.astype(np.float16).view(np.uint16)) or \
            np.max(np.abs(out16.astype(np.float64) - ref)) <= 2.0 ** -11 * np.max(np.abs(ref))


def pin_closed_forms(lib, seed=12):
    rng = np.random.default_rng(seed)
    H, Hk, d, bs = 4, 2, 64, 16
    scale = 0.125
    # one token: p = 1, out = V_0 exactly, lse = s_0
    q, K, V, lens = logical_problem(rng, 2, H, Hk, d, (1, 1))
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    out, lse, _ = run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, bs)
    for b in range(2):
        for h in range(H):
            assert np.array_equal(out[b, h], V[b, h // 2, 0].astype(np.float64))
            s0 = scale * float(np.dot(q[b, h].astype(np.float64), K[b, h // 2, 0].astype(np.float64)))
            assert abs(lse[b, h] - s0) <= 1e-12
    # zero query: uniform weights, out = mean of V, lse = ln L
    q0 = np.zeros_like(q)
    q_, K, V, lens = logical_problem(rng, 2, H, Hk, d, (37, 5))
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    out, lse, _ = run_decode(lib, q0, kc, vc, bt, lens, scale, H, Hk, d, bs)
    for b, L in enumerate(lens):
        for h in range(H):
            mean = V[b, h // 2, :L].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(out[b, h] - mean)) <= 1e-14
            assert abs(lse[b, h] - math.log(L)) <= 1e-14
    # equal keys: uniform weights again, with a nonzero query
    Keq = np.repeat(K[:, :, :1, :], K.shape[2], axis=2)
    kc, vc, bt = paginate(Keq, V, lens, bs, rng)
    out, _, _ = run_decode(lib, q_, kc, vc, bt, lens, scale, H, Hk, d, bs)
    for b, L in enumerate(lens):
        for h in range(H):
            mean = V[b, h // 2, :L].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(out[b, h] - mean)) <= 1e-14
    # two tokens, logits 0 and 2*scale: out = (V0 + e^(2 scale) V1) / (1 + e^(2 scale))
    q2 = np.zeros((1, H, d), dtype=np.float16)
    q2[0, :, 3] = 1.0
    K2 = np.zeros((1, Hk, 2, d), dtype=np.float16)
    K2[0, :, 1, 3] = 2.0
    V2 = randn16(rng, (1, Hk, 2, d))
    kc, vc, bt = paginate(K2, V2, (2,), bs, rng)
    out, lse, _ = run_decode(lib, q2, kc, vc, bt, (2,), scale, H, Hk, d, bs)
    w = math.exp(2 * scale)
    for h in range(H):
        v0 = V2[0, h // 2, 0].astype(np.float64)
        v1 = V2[0, h // 2, 1].astype(np.float64)
        assert np.max(np.abs(out[0, h] - (v0 + w * v1) / (1 + w))) <= 1e-15
        assert abs(lse[0, h] - math.log(1 + w)) <= 1e-15
    # a dominant logit: out = V at the argmax
    q, K, V, lens = logical_problem(rng, 2, H, Hk, d, (29, 50))
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    out, _, _ = run_decode(lib, q, kc, vc, bt, lens, 1e4, H, Hk, d, bs)
    for b, L in enumerate(lens):
        for h in range(H):
            s = K[b, h // 2, :L].astype(np.float64) @ q[b, h].astype(np.float64)
            top = np.sort(s)[-2:]
            if top[1] - top[0] < 1e-3:
                continue
            assert np.array_equal(out[b, h], V[b, h // 2, int(np.argmax(s))].astype(np.float64))
    # all-ones values: the weights sum to one
    q, K, V, lens = logical_problem(rng, 3, H, Hk, d, (64, 3, 19))
    ones = np.ones_like(V)
    kc, vc, bt = paginate(K, ones, lens, bs, rng)
    out, _, _ = run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, bs)
    assert np.max(np.abs(out - 1.0)) <= 1e-14
    # empty sequence: out = 0, lse = -inf
    q, K, V, _ = logical_problem(rng, 2, H, Hk, d, (4, 4))
    lens = np.array([0, 4])
    kc, vc, bt = paginate(K, V, np.array([1, 4]), bs, rng)
    out, lse, _ = run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, bs)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))


def pin_invariances(lib, seed=13):
    rng = np.random.default_rng(seed)
    H, Hk, d = 8, 2, 64
    scale = 1.0 / 8.0
    q, K, V, lens = logical_problem(rng, 3, H, Hk, d, (70, 16, 33))
    # physical block order
    kc, vc, bt = paginate(K, V, lens, 16, rng)
    ref, ref_lse, _ = run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, 16)
    kc2, vc2, bt2 = paginate(K, V, lens, 16, rng)
    out, lse, _ = run_decode(lib, q, kc2, vc2, bt2, lens, scale, H, Hk, d, 16)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
    # block size 1 vs 16 holding the same logical K/V
    kc1, vc1, bt1 = paginate(K, V, lens, 1, rng)
    out, lse, _ = run_decode(lib, q, kc1, vc1, bt1, lens, scale, H, Hk, d, 1)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
    # shared prefix blocks vs copied blocks
    Ks, Vs = K.copy(), V.copy()
    Ks[1:, :, :32] = Ks[0, :, :32]
    Vs[1:, :, :32] = Vs[0, :, :32]
    lens_s = np.array([70, 40, 33])
    kc, vc, bt = paginate(Ks, Vs, lens_s, 16, rng)
    copied, copied_lse, _ = run_decode(lib, q, kc, vc, bt, lens_s, scale, H, Hk, d, 16)
    kc, vc, bt = paginate(Ks, Vs, lens_s, 16, rng, shared=([0, 1, 2], 2))
    assert len(set(bt[:, 0])) == 1 and len(set(bt[:, 1])) == 1
    out, lse, _ = run_decode(lib, q, kc, vc, bt, lens_s, scale, H, Hk, d, 16)
    assert np.array_equal(out, copied) and np.array_equal(lse, copied_lse)
    # GQA equals MHA with each KV head replicated g times
    g = H // Hk
    Kr = np.repeat(K, g, axis=1)
    Vr = np.repeat(V, g, axis=1)
    kcm, vcm, btm = paginate(Kr, Vr, lens, 16, rng)
    out, lse, _ = run_decode(lib, q, kcm, vcm, btm, lens, scale, H, H, d, 16)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def pin_merge(lib, seed=14):
    """Partials over any split of [0, L) merge back to the full result."""
    rng = np.random.default_rng(seed)
    H, Hk, d, bs = 4, 1, 64, 16
    scale = 0.2
    q, K, V, lens = logical_problem(rng, 1, H, Hk, d, (150,))
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    full, full_lse, _ = run_decode(lib, q, kc, vc, bt, lens, scale, H, Hk, d, bs)
    for cuts in ([0, 150], [0, 16, 150], [0, 1, 2, 64, 149, 150], [0, 75, 75, 150]):
        for h in range(H):
            parts = [oracle.partial(q, kc, vc, bt, scale, H, Hk, d, bs, 0, h, a, z, lib=lib)
                     for a, z in zip(cuts[:-1], cuts[1:])]
            m = np.array([p[0] for p in parts])
            l = np.array([p[1] for p in parts])
            acc = np.stack([p[2] for p in parts])
            out, lse = oracle.lse_merge(m, l, acc, lib=lib)
            assert np.max(np.abs(out - full[0, h])) <= 1e-12
            assert abs(lse - full_lse[0, h]) <= 1e-12
            # each partial against its own closed form
            for (a, z), (pm, pl, pacc) in zip(zip(cuts[:-1], cuts[1:]), parts):
                if z == a:
                    assert pm == -np.inf and pl == 0.0 and not pacc.any()
                    continue
                s = scale * (K[0, 0, a:z].astype(np.float64) @ q[0, h].astype(np.float64))
                assert abs(pm - s.max()) <= 1e-12
                w = np.exp(s - s.max())
                assert abs(pl - w.sum()) <= 1e-12 * max(1.0, w.sum())
                assert np.max(np.abs(pacc - w @ V[0, 0, a:z].astype(np.float64))) <= 1e-11
    # two hand-made partials: weights e^(m_i - M) l_i
    m = np.array([0.0, math.log(3.0)])
    l = np.array([1.0, 1.0])
    acc = np.array([[2.0] * 4, [6.0] * 4])
    out, lse = oracle.lse_merge(m, l, acc, lib=lib)
    # M = ln 3: weights 1/3 and 1 -> out = (2/3 + 6) / (1/3 + 1) = 5
    assert np.allclose(out, 5.0, rtol=0, atol=1e-14) and abs(lse - math.log(4.0)) <= 1e-14


def pin_poison(lib, seed=15):
    """Rows, blocks and table entries outside [0, L) are never read."""
    rng = np.random.default_rng(seed)
    H, Hk, d, bs = 4, 2, 64, 16
    q, K, V, lens = logical_problem(rng, 3, H, Hk, d, (17, 32, 5))
    kc, vc, bt = paginate(K, V, lens, bs, rng, poison=False, extra_blocks=4)
    clean, clean_lse, _ = run_decode(lib, q, kc, vc, bt, lens, 0.125, H, Hk, d, bs)
    kc2, vc2, bt2 = paginate(K, V, lens, bs, rng, poison=True, extra_blocks=4)
    bt2 = np.concatenate([bt2, np.full((3, 2), -99, dtype=np.int32)], axis=1)
    out, lse, _ = run_decode(lib, q, kc2, vc2, bt2, lens, 0.125, H, Hk, d, bs)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out, clean) and np.array_equal(lse, clean_lse)


def pin_append(lib, seed=16):
    """Append scatter equals numpy fancy-index assignment; -1 slots skipped."""
    rng = np.random.default_rng(seed)
    NB, Hk, bs, d = 9, 3, 16, 64
    kc = randn16(rng, (NB, Hk, bs, d))
    vc = randn16(rng, (NB, Hk, bs, d))
    T = 20
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[[2, 11]] = -1
    kn = randn16(rng, (T, Hk, d))
    vn = randn16(rng, (T, Hk, d))
    k2, v2 = oracle.append(kn, vn, slots, kc, vc, bs, lib=lib)
    keep = slots >= 0
    for cache, new, got in ((kc, kn, k2), (vc, vn, v2)):
        ref = cache.copy()
        flat = ref.transpose(0, 2, 1, 3).reshape(NB * bs, Hk, d).copy()
        flat[slots[keep]] = new[keep]
        ref = flat.reshape(NB, bs, Hk, d).transpose(0, 2, 1, 3)
        assert np.array_equal(got.view(np.uint16), np.ascontiguousarray(ref).view(np.uint16))
    bad = slots.copy()
    bad[0] = NB * bs
    try:
        oracle.append(kn, vn, bad, kc, vc, bs, lib=lib)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("slot beyond the pool accepted")


def pin_append_then_attend(lib, seed=17):
    """Appending token L-1 by slot, then attending, equals dense attention
    over the logical sequence that ends with that token."""
    rng = np.random.default_rng(seed)
    H, Hk, d, bs = 4, 2, 64, 16
    q, K, V, lens = logical_problem(rng, 3, H, Hk, d, (16, 17, 1))
    pre = lens - 1
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    # forget the last token of each sequence, then append it by slot
    for b, L in enumerate(lens):
        t = int(L) - 1
        kc[bt[b, t // bs], :, t % bs] = np.float16(np.nan)
        vc[bt[b, t // bs], :, t % bs] = np.float16(np.nan)
    kn = np.stack([K[b, :, int(L) - 1] for b, L in enumerate(lens)])
    vn = np.stack([V[b, :, int(L) - 1] for b, L in enumerate(lens)])
    slots = np.array([int(bt[b, int(L - 1) // bs]) * bs + int(L - 1) % bs
                      for b, L in enumerate(lens)], dtype=np.int64)
    kc2, vc2 = oracle.append(kn, vn, slots, kc, vc, bs, lib=lib)
    out, lse, _ = run_decode(lib, q, kc2, vc2, bt, lens, 0.125, H, Hk, d, bs)
    ref, ref_lse = dense_reference(q, K, V, lens, 0.125, H, Hk)
    assert np.max(np.abs(out - ref)) <= 1e-12 and np.max(np.abs(lse - ref_lse)) <= 1e-12
    assert pre.min() == 0


def pin_rejects_bad_input(lib, seed=18):
    rng = np.random.default_rng(seed)
    H, Hk, d, bs = 4, 2, 64, 16
    q, K, V, lens = logical_problem(rng, 2, H, Hk, d, (20, 3))
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    for bad in ("block", "len"):
        bt2, lens2 = bt.copy(), lens.copy()
        if bad == "block":
            bt2[0, 1] = kc.shape[0]
        else:
            lens2[1] = bt.shape[1] * bs + 1
        try:
            run_decode(lib, q, kc, vc, bt2, lens2, 0.125, H, Hk, d, bs)
        except oracle.OracleError:
            continue
        raise AssertionError(f"bad {bad} accepted")


# ----------------------------------------------------------------------------
# FP8 (E4M3) KV cache pins: torch's float8_e4m3fn conversions are the
# independent library routine (they round to nearest-even but turn overflow
# into NaN, so the saturation of the library's reading is pinned by closed
# forms instead)
# ----------------------------------------------------------------------------

def _torch_e4m3_codes(y32):
    """torch's E4M3 codes of fp32 values already inside [-448, 448]."""
    t = torch.from_numpy(np.ascontiguousarray(y32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_e4m3_values(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_decode(lib):
    codes = np.arange(256, dtype=np.uint8)
    ref = _torch_e4m3_values(codes)
    got = np.array([lib.pkvo_e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def pin_e4m3_encode(lib, seed=21):
    rng = np.random.default_rng(seed)
    codes = np.arange(256, dtype=np.uint8)
    vals = _torch_e4m3_values(codes)
    finite = ~np.isnan(vals)
    # every code round-trips (both zeros included)
    back = oracle.f32_to_e4m3(vals[finite].astype(np.float32), lib=lib)
    assert np.array_equal(back, codes[finite])
    # midpoints between neighbours, and random values, against torch (in range)
    pos = np.sort(np.unique(np.abs(vals[finite])))
    mids = (pos[:-1] + pos[1:]) / 2.0
    ys = np.concatenate([mids, -mids, rng.uniform(-447.0, 447.0, 20000),
                         rng.standard_normal(20000) * 10.0 ** rng.integers(-4, 2, 20000)])
    ys = ys.astype(np.float32)
    ys = ys[np.abs(ys) < 448.0]
    got = oracle.f32_to_e4m3(ys, lib=lib)
    ref = _torch_e4m3_codes(ys)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(ys[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]
    # closed forms of the saturating reading: finite overflow and infinities
    # go to +-448, NaN to the NaN code
    sat = np.array([448.0, 455.0, 463.9, 464.0, 480.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(oracle.f32_to_e4m3(sat, lib=lib) == 0x7E)
    assert np.all(oracle.f32_to_e4m3(-sat, lib=lib) == 0xFE)
    assert oracle.f32_to_e4m3(np.array([np.nan], dtype=np.float32), lib=lib)[0] == 0x7F
    tiny = np.array([2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -9, 2.0 ** -11], dtype=np.float32)
    assert list(oracle.f32_to_e4m3(tiny, lib=lib)) == [0x00, 0x02, 0x01, 0x00]


def pin_e4m3_quantize(lib):
    """Every finite fp16 value under several scales: E4M3(fp32(x) / fp32(s)),
    the quotient by numpy's IEEE fp32 division, the rounding by torch."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x16 = bits.view(np.float16)
    ok = np.isfinite(x16)
    bits, x16 = bits[ok], x16[ok]
    for s in (1.0, 0.0123, 3.5, 1.0 / 64, 448.0 / 65504.0):
        s32 = np.float32(s)
        y = x16.astype(np.float32) / s32
        got = oracle.quantize_e4m3(bits, s32, lib=lib)
        inr = np.abs(y) < 448.0
        ref = np.where(y >= 0, 0x7E, 0xFE).astype(np.uint8)
        ref[inr] = _torch_e4m3_codes(y[inr])
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, (s, [(float(x16[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]])
    inf = np.array([0x7C00, 0xFC00], dtype=np.uint16)
    assert list(oracle.quantize_e4m3(inf, 1.0, lib=lib)) == [0x7E, 0xFE]


def _paginate_codes(K8, V8, lens, bs, rng, poison=True):
    """paginate() for uint8 code arrays (poison: the NaN code 0x7f)."""
    kc16, vc16, bt = paginate(K8.astype(np.float16), V8.astype(np.float16), lens, bs, rng,
                              poison=poison)
    # codes 0..255 are exact in fp16 and NaN marks the poisoned rows
    kc = np.where(np.isnan(kc16), 0x7F, kc16).astype(np.uint8)
    vc = np.where(np.isnan(vc16), 0x7F, vc16).astype(np.uint8)
    return kc, vc, bt


def pin_f8_dense(lib, seed=22):
    """FP8 paged attention = float64 SDPA over torch-dequantized K/V."""
    rng = np.random.default_rng(seed)
    for (B, H, Hk, d, bs, lens, ks, vs) in [(3, 4, 2, 64, 16, (1, 17, 40), 0.02, 0.015),
                                            (2, 8, 1, 128, 16, (33, 16), 1.0, 0.5),
                                            (2, 8, 2, 64, 8, (15, 64), 0.003, 2.0)]:
        q = randn16(rng, (B, H, d))
        Lmax = max(lens)
        K8 = rng.integers(0, 256, (B, Hk, Lmax, d)).astype(np.uint8)
        V8 = rng.integers(0, 256, (B, Hk, Lmax, d)).astype(np.uint8)
        K8[(K8 & 0x7F) == 0x7F] = 0x3C   # no NaN codes in attended rows
        V8[(V8 & 0x7F) == 0x7F] = 0x41
        kc, vc, bt = _paginate_codes(K8, V8, lens, bs, rng)
        scale = 1.0 / math.sqrt(d)
        out, lse = oracle.decode_f8(q, kc, vc, ks, vs, bt, np.asarray(lens, np.int32), scale,
                                    H, Hk, d, bs, lib=lib)
        Kd = _torch_e4m3_values(K8) * float(np.float32(ks))
        Vd = _torch_e4m3_values(V8) * float(np.float32(vs))
        ref, ref_lse = dense_reference(q, Kd, Vd, lens, scale, H, Hk)
        assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
        assert np.max(np.abs(lse - ref_lse)) <= 1e-12 * max(1.0, np.max(np.abs(ref_lse)))


def pin_f8_append(lib, seed=23):
    """FP8 append = torch quantization (clamped to +-448 first) scattered by
    numpy fancy indexing; -1 slots skipped; other bytes untouched."""
    rng = np.random.default_rng(seed)
    NB, Hk, bs, d = 7, 2, 16, 64
    kc = rng.integers(0, 256, (NB, Hk, bs, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (NB, Hk, bs, d)).astype(np.uint8)
    T = 12
    slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
    slots[[3, 7]] = -1
    kn = (rng.standard_normal((T, Hk, d)) * 40.0).astype(np.float16)
    vn = randn16(rng, (T, Hk, d))
    ks, vs = np.float32(0.05), np.float32(0.011)
    k2, v2 = oracle.append_f8(kn, vn, slots, kc, vc, bs, ks, vs, lib=lib)
    keep = slots >= 0
    for cache, new, s, got in ((kc, kn, ks, k2), (vc, vn, vs, v2)):
        y = np.clip(new.astype(np.float32) / s, -448.0, 448.0)
        codes = _torch_e4m3_codes(y)
        ref = cache.copy()
        flat = ref.transpose(0, 2, 1, 3).reshape(NB * bs, Hk, d).copy()
        flat[slots[keep]] = codes[keep]
        ref = flat.reshape(NB, bs, Hk, d).transpose(0, 2, 1, 3)
        assert np.array_equal(got, np.ascontiguousarray(ref))
    assert np.any(np.abs(kn.astype(np.float32) / ks) > 448.0)  # saturation exercised


def pin_f8_poison(lib, seed=24):
    """NaN codes in unread rows, blocks and table entries change no output bit."""
    rng = np.random.default_rng(seed)
    B, H, Hk, d, bs, lens = 3, 4, 2, 64, 16, (17, 32, 5)
    q = randn16(rng, (B, H, d))
    K8 = rng.integers(0, 0x70, (B, Hk, max(lens), d)).astype(np.uint8)
    V8 = rng.integers(0x80, 0xF0, (B, Hk, max(lens), d)).astype(np.uint8)
    kc, vc, bt = _paginate_codes(K8, V8, lens, bs, np.random.default_rng(1), poison=False)
    kc2, vc2, bt2 = _paginate_codes(K8, V8, lens, bs, np.random.default_rng(1), poison=True)
    assert np.any(kc2 == 0x7F)
    a = oracle.decode_f8(q, kc, vc, 0.1, 0.2, bt, np.asarray(lens, np.int32), 0.125, H, Hk, d,
                         bs, lib=lib)
    b = oracle.decode_f8(q, kc2, vc2, 0.1, 0.2, bt2, np.asarray(lens, np.int32), 0.125, H, Hk,
                         d, bs, lib=lib)
    assert np.all(np.isfinite(a[0])) and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ----------------------------------------------------------------------------
# multi-token (causal) paged attention pins
# ----------------------------------------------------------------------------

def multi_problem(rng, B, H, Hk, d, lens, nq):
    """Logical K/V [B, Hk, Lmax, d] and packed queries [sum(nq), H, d]."""
    lens = np.asarray(lens)
    K = randn16(rng, (B, Hk, int(lens.max()), d))
    V = randn16(rng, (B, Hk, int(lens.max()), d))
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = randn16(rng, (int(qs[-1]), H, d))
    return q, K, V, lens, qs


def dense_causal_reference(q, K, V, lens, qs, scale, H, Hk):
    """float64 torch SDPA with an explicit causal mask aligned to the end of
    each sequence, and scipy's logsumexp over the same masked logits."""
    TQ, _, d = q.shape
    g = H // Hk
    out = np.zeros((TQ, H, d))
    lse = np.full((TQ, H), -np.inf)
    for b in range(len(lens)):
        L = int(lens[b])
        r0, r1 = int(qs[b]), int(qs[b + 1])
        n = r1 - r0
        if n == 0:
            continue
        qt = torch.from_numpy(q[r0:r1].astype(np.float64)).permute(1, 0, 2).reshape(1, H, n, d)
        kt = torch.from_numpy(K[b, :, :L].astype(np.float64)).repeat_interleave(g, dim=0)
        vt = torch.from_numpy(V[b, :, :L].astype(np.float64)).repeat_interleave(g, dim=0)
        pos = np.arange(n)[:, None] + (L - n)
        allowed = np.arange(L)[None, :] <= pos
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.reshape(1, H, L, d), vt.reshape(1, H, L, d),
            attn_mask=torch.from_numpy(allowed), scale=scale)
        out[r0:r1] = o.reshape(H, n, d).permute(1, 0, 2).numpy()
        s = np.einsum("nhd,hld->nhl", q[r0:r1].astype(np.float64), kt.numpy()) * scale
        s = np.where(allowed[:, None, :], s, -np.inf)
        lse[r0:r1] = scipy.special.logsumexp(s, axis=2)
    return out, lse


def pin_multi_dense(lib, seed=31):
    """Multi-token paged attention = causal float64 SDPA on contiguous K/V."""
    rng = np.random.default_rng(seed)
    for (B, H, Hk, d, bs, lens, nq) in [(3, 4, 2, 64, 16, (5, 17, 40), (1, 4, 8)),
                                        (2, 8, 2, 128, 16, (33, 16), (16, 3)),
                                        (3, 4, 4, 64, 1, (9, 3, 6), (2, 3, 0)),
                                        (2, 8, 1, 64, 8, (64, 20), (5, 20))]:
        q, K, V, lens, qs = multi_problem(rng, B, H, Hk, d, lens, nq)
        scale = 1.0 / math.sqrt(d)
        kc, vc, bt = paginate(K, V, lens, bs, rng)
        out, lse = oracle.decode_multi(q, kc, vc, bt, lens.astype(np.int32), qs, scale, H, Hk,
                                       d, bs, lib=lib)
        ref, ref_lse = dense_causal_reference(q, K, V, lens, qs, scale, H, Hk)
        assert np.max(np.abs(out - ref)) <= 1e-12, np.max(np.abs(out - ref))
        assert np.max(np.abs(lse - ref_lse)) <= 1e-12


def pin_multi_is_truncated_decode(lib, seed=32):
    """Query token i of a sequence equals a one-token decode of the same query
    over the context cut at its position (bitwise); one query per sequence is
    exactly the decode."""
    rng = np.random.default_rng(seed)
    B, H, Hk, d, bs = 3, 4, 2, 64, 16
    q, K, V, lens, qs = multi_problem(rng, B, H, Hk, d, (12, 33, 7), (3, 5, 7))
    kc, vc, bt = paginate(K, V, lens, bs, rng)
    out, lse = oracle.decode_multi(q, kc, vc, bt, lens.astype(np.int32), qs, 0.125, H, Hk, d,
                                   bs, lib=lib)
    for b in range(B):
        n = int(qs[b + 1] - qs[b])
        for i in range(n):
            cut = lens.copy()
            cut[b] = lens[b] - n + i + 1
            qd = np.repeat(q[qs[b] + i][None], B, axis=0)
            o1, l1, _ = run_decode(lib, qd, kc, vc, bt, cut, 0.125, H, Hk, d, bs)
            assert np.array_equal(out[qs[b] + i], o1[b]) and np.array_equal(lse[qs[b] + i], l1[b])
    ones = np.arange(B + 1, dtype=np.int32)
    q1 = q[:B]
    o_m, l_m = oracle.decode_multi(q1, kc, vc, bt, lens.astype(np.int32), ones, 0.125, H, Hk, d,
                                   bs, lib=lib)
    o_d, l_d, _ = run_decode(lib, q1, kc, vc, bt, lens, 0.125, H, Hk, d, bs)
    assert np.array_equal(o_m, o_d) and np.array_equal(l_m, l_d)


def pin_multi_poison_and_rejects(lib, seed=33):
    rng = np.random.default_rng(seed)
    B, H, Hk, d, bs = 2, 4, 2, 64, 16
    q, K, V, lens, qs = multi_problem(rng, B, H, Hk, d, (17, 30), (4, 2))
    kc, vc, bt = paginate(K, V, lens, bs, np.random.default_rng(2), poison=False)
    kc2, vc2, bt2 = paginate(K, V, lens, bs, np.random.default_rng(2), poison=True)
    a = oracle.decode_multi(q, kc, vc, bt, lens.astype(np.int32), qs, 0.125, H, Hk, d, bs,
                            lib=lib)
    b = oracle.decode_multi(q, kc2, vc2, bt2, lens.astype(np.int32), qs, 0.125, H, Hk, d, bs,
                            lib=lib)
    assert np.all(np.isfinite(a[0])) and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    bad = lens.copy()
    bad[0] = 3  # fewer cached tokens than query tokens
    try:
        oracle.decode_multi(q, kc, vc, bt, bad.astype(np.int32), qs, 0.125, H, Hk, d, bs, lib=lib)
    except oracle.OracleError:
        pass
    else:
        raise AssertionError("more query tokens than context accepted")


ALL_PINS = [pin_fp16_decode, pin_fp16_encode, pin_dense_sdpa, pin_closed_forms,
            pin_invariances, pin_merge, pin_poison, pin_append, pin_append_then_attend,
            pin_rejects_bad_input, pin_e4m3_decode, pin_e4m3_encode, pin_e4m3_quantize,
            pin_f8_dense, pin_f8_append, pin_f8_poison, pin_multi_dense,
            pin_multi_is_truncated_decode, pin_multi_poison_and_rejects]
