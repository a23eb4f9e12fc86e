"""The C-ABI library builds for sm_103a, loads, exports every function
include/pagedkv.h declares, and rejects bad arguments on the host (these
calls return before any CUDA work, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_213_gb300 as pkv
from paged_kv_cache_213_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.library()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"paged_kv_append", "paged_decode_attention", "paged_decode_plan",
            "paged_kv_get_error", "paged_kv_status_string"} <= set(names)
    raw = ctypes.CDLL(pkv.library_path())
    for n in names:
        assert hasattr(raw, n), f"{n} not exported"


def header_defines():
    """Integer #defines of include/pagedkv.h, by name."""
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    out = {}
    for name, expr in re.findall(r"^#define\s+(PKV_\w+)\s+([(0-9][^/\n]*)", text, flags=re.M):
        expr = re.sub(r"(\d)u\b", r"\1", expr.strip())
        assert re.fullmatch(r"[0-9a-fA-Fx()<\s]+", expr), expr
        out[name] = int(eval(expr))  # digits, parentheses and shifts only
    return out


def test_python_constants_match_the_header():
    d = header_defines()
    for name in ("PKV_ERRBIT_BLOCK_ID", "PKV_ERRBIT_SLOT", "PKV_ERRBIT_CONTEXT",
                 "PKV_ERRBIT_TIMEOUT", "PKV_ERRBIT_WORKSPACE", "PKV_ERRBIT_APPEND",
                 "PKV_TABLES_READY", "PKV_APPEND_NEWEST", "PKV_WORKSPACE_COUNTER_BYTES"):
        assert getattr(pkv, name) == d[name], name
    bits = [d[n] for n in d if n.startswith("PKV_ERRBIT_")]
    assert len(bits) == 6 and sum(bits) == 0x3f  # distinct single bits
    assert d["PKV_TABLES_READY"] & d["PKV_APPEND_NEWEST"] == 0
    assert d["PKV_NOALLOC_SCRATCH_BYTES"] == 16 << 20
    assert d["PKV_WORKSPACE_COUNTER_BYTES"] < d["PKV_NOALLOC_SCRATCH_BYTES"]


def test_copy_in_host_checks(lib):
    """Zero bytes is a no-op; NULL, misaligned or ragged copies are rejected,
    all before any CUDA call."""
    fn = lib.paged_copy_in
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(None, None, 0, None) == 0
    assert fn(None, ctypes.c_void_p(4096), 64, None) == -1
    assert fn(ctypes.c_void_p(4096), ctypes.c_void_p(4104), 64, None) == -1  # misaligned
    assert fn(ctypes.c_void_p(4096), ctypes.c_void_p(8192), 40, None) == -1  # not 16n bytes


def test_workspace_clear_host_checks(lib):
    """Zero bytes is a no-op and a NULL workspace with bytes is rejected, both
    before any CUDA call."""
    assert lib.paged_decode_workspace_clear(None, 0, None) == 0
    assert lib.paged_decode_workspace_clear(None, 4096, None) == -1


def test_status_strings(lib):
    assert pkv.status_string(0) == "ok"
    for s in (-1, -2, -3, -4, -5):
        assert pkv.status_string(s) not in ("ok", "unknown status")
    assert pkv.status_string(42) == "unknown status"


def _plan(lib, *args):
    P = ctypes.c_int(-1)
    W = ctypes.c_size_t(0)
    rc = lib.paged_decode_plan(*args, ctypes.byref(P), ctypes.byref(W))
    return rc, P.value, W.value


def test_plan_explicit_partition(lib):
    # B=32, H=32, Hk=8, d=128, bs=16, MB=128, max_len 2048, P=256 -> 8 partitions
    rc, P, W = _plan(lib, 32, 32, 8, 128, 16, 128, 2048, 256)
    assert rc == 0 and P == 256
    rows = 32 * 32 * 8
    up = lambda x: (x + 255) // 256 * 256
    assert W == up(rows * 128 * 4) + 2 * up(rows * 4)
    # one partition covers everything: no workspace
    rc, P, W = _plan(lib, 32, 32, 8, 128, 16, 128, 256, 256)
    assert rc == 0 and W == 0
    # max_context_len <= 0 means MB * bs
    rc, P, W = _plan(lib, 2, 8, 2, 64, 16, 4, 0, 16)
    assert rc == 0 and W == up(2 * 8 * 4 * 64 * 4) + 2 * up(2 * 8 * 4 * 4)


@pytest.mark.parametrize("args,status", [
    ((4, 6, 4, 128, 16, 8, 0, 64), -1),    # 6 % 4 != 0
    ((4, 8, 2, 96, 16, 8, 0, 64), -2),     # head_dim 96 not built
    ((4, 8, 2, 128, 12, 8, 0, 48), -2),    # block size 12
    ((4, 48, 2, 128, 16, 8, 0, 64), -2),   # group 24
    ((4, 8, 2, 128, 16, 8, 0, 24), -1),    # partition not a multiple of 16
    ((4, 8, 2, 128, 32, 8, 0, 16), -1),    # partition not a multiple of the block size
    ((4, 8, 2, 128, 1, 8, 0, 4096), -1),   # more than 2048 blocks per partition
    ((-1, 8, 2, 128, 16, 8, 0, 64), -1),
    ((4, 8, 2, 128, 16, 0, 0, 64), -1),
])
def test_plan_rejects(lib, args, status):
    assert _plan(lib, *args)[0] == status


def test_calls_reject_bad_arguments_without_launching(lib):
    n = None
    # append: zero tokens is a no-op, null pointers and odd head_dim are errors
    assert lib.paged_kv_append(n, n, n, n, n, 0, 8, 128, 16, 10, n, n) == 0
    assert lib.paged_kv_append(n, n, n, n, n, 4, 8, 128, 16, 10, n, n) == -1
    assert lib.paged_kv_append(n, n, n, n, n, 4, 8, 100, 16, 10, n, n) == -1
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.paged_kv_append(fake, odd, fake, fake, fake, 4, 8, 128, 16, 10, n, n) == -1
    # attention: null pointers, misalignment, missing workspace
    args = dict(B=4, MB=8, NB=40, H=8, Hk=2, d=128, bs=16)

    def call(out, q, kc, vc, bt, cl, mcl=0, P=64, ws=None, ws_bytes=0, scale=0.1):
        return lib.paged_decode_attention(out, q, kc, vc, bt, cl, args["B"], args["MB"],
                                          args["NB"], scale, args["H"], args["Hk"], args["d"],
                                          args["bs"], mcl, P, ws, ws_bytes, n, n, n)
    assert call(n, fake, fake, fake, fake, fake) == -1
    assert call(odd, fake, fake, fake, fake, fake) == -1
    assert call(fake, fake, fake, fake, fake, fake) == -3          # 2 partitions, no workspace
    assert call(fake, fake, fake, fake, fake, fake, ws=fake, ws_bytes=64) == -3
    assert call(fake, fake, fake, fake, fake, fake, scale=float("nan")) == -1
    assert lib.paged_kv_get_error(n, n, n) == -1
    # the flagged call: the same checks, and unknown flag bits are rejected first

    def call_ex(flags, out=fake, ws=None):
        return lib.paged_decode_attention_ex(out, fake, fake, fake, fake, fake, args["B"],
                                             args["MB"], args["NB"], 0.1, args["H"], args["Hk"],
                                             args["d"], args["bs"], 0, 64, ws, 0, n, n, n, flags)
    assert call_ex(0x2) == -1 and call_ex(0xffff0000) == -1
    assert call_ex(pkv.PKV_TABLES_READY, out=n) == -1
    assert call_ex(pkv.PKV_TABLES_READY) == -3                     # no workspace
    # every _ex entry point rejects unknown flag bits before anything else
    c = ctypes
    p_ = c.c_void_p
    f8 = lib.paged_decode_attention_fp8_ex
    f8.argtypes = [p_] * 6 + [c.c_int, c.c_int, c.c_int64, c.c_float, c.c_float, c.c_float] + \
        [c.c_int] * 5 + [p_, c.c_size_t, p_, p_, p_, c.c_uint32]
    f8.restype = c.c_int
    assert f8(fake, fake, fake, fake, fake, fake, 4, 8, 40, 0.1, 1.0, 1.0, 8, 2, 128, 16, 0,
              fake, 1 << 20, n, n, n, 0x10) == -1
    mu = lib.paged_decode_attention_multi_ex
    mu.argtypes = [p_] * 7 + [c.c_int] * 4 + [c.c_int64, c.c_float] + [c.c_int] * 6 + \
        [p_, c.c_size_t, p_, p_, p_, c.c_uint32]
    mu.restype = c.c_int
    assert mu(fake, fake, fake, fake, fake, fake, fake, 4, 8, 2, 8, 40, 0.1, 8, 2, 128, 16, 0,
              0, fake, 1 << 20, n, n, n, 0x10) == -1
    st = lib.paged_decode_step_ex
    st.argtypes = [p_, p_, p_, c.c_int] + [p_] * 6 + [c.c_int, c.c_int, c.c_int64, c.c_float] + \
        [c.c_int] * 6 + [p_, c.c_size_t, p_, p_, p_, c.c_uint32]
    st.restype = c.c_int
    for bad in (0x4, 0x10, 0x80000000):
        assert st(fake, fake, fake, 4, fake, fake, fake, fake, fake, fake, 4, 8, 40, 0.1, 8, 2,
                  128, 16, 0, 0, fake, 1 << 20, n, n, n, bad) == -1


def test_step_launches_with_fixed_partitions(lib):
    """The launch count of a step, for plans that need no device query: the
    append, then one kernel (one partition) or two (partitions + merge)."""
    # B=4, 8/2 heads, d=128, bs=16, 8 blocks per sequence: up to 128 tokens
    assert pkv.step_launches(4, 8, 2, 128, 16, 8, 0, 64) == 3
    assert pkv.step_launches(4, 8, 2, 128, 16, 8, 0, 128) == 2
    assert pkv.step_launches(4, 8, 2, 128, 16, 8, 0, 64, num_tokens=0) == 2
    # the fused append needs the balanced split: fixed partitions keep the append
    assert pkv.step_launches(4, 8, 2, 128, 16, 8, 0, 128, flags=pkv.PKV_APPEND_NEWEST) == 2
    with pytest.raises(pkv.PagedKVError):
        pkv.step_launches(4, 8, 2, 128, 16, 8, 0, 128, flags=0x8)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="a GPU is present")
def test_auto_plan_needs_a_device(lib):
    rc, _, _ = _plan(lib, 4, 8, 2, 128, 16, 8, 0, 0)
    assert rc == -4


def test_fp8_host_rejections(lib):
    import ctypes as c
    p = c.c_void_p
    fn = lib.paged_kv_append_fp8
    fn.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64, c.c_float,
                   c.c_float, p, p]
    fn.restype = c.c_int
    x = p(256)
    # head_dim not a multiple of 16, a zero scale, a NaN scale: rejected before any launch
    assert fn(x, x, x, x, x, 4, 2, 8, 16, 10, 1.0, 1.0, None, None) == -1
    assert fn(x, x, x, x, x, 4, 2, 64, 16, 10, 0.0, 1.0, None, None) == -1
    assert fn(x, x, x, x, x, 4, 2, 64, 16, 10, 1.0, float("nan"), None, None) == -1
    att = lib.paged_decode_attention_fp8
    att.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float, c.c_float,
                    c.c_float, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p, c.c_size_t, p, p,
                    p]
    att.restype = c.c_int
    assert att(x, x, x, x, x, x, 4, 8, 10, 0.1, -1.0, 1.0, 8, 2, 128, 16, 0, x, 1 << 20, None,
               None, None) == -1


def _multi_fns(lib):
    c = ctypes
    p = c.c_void_p
    plan = lib.paged_decode_multi_plan
    plan.argtypes = [c.c_int] * 10 + [c.POINTER(c.c_int), c.POINTER(c.c_size_t)]
    plan.restype = c.c_int
    att = lib.paged_decode_attention_multi
    att.argtypes = [p, p, p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int64,
                    c.c_float, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int, p,
                    c.c_size_t, p, p, p]
    att.restype = c.c_int
    return plan, att


def _multi_plan(plan, *args):
    P = ctypes.c_int(-1)
    W = ctypes.c_size_t(0)
    rc = plan(*args, ctypes.byref(P), ctypes.byref(W))
    return rc, P.value, W.value


def test_multi_plan_explicit_partition(lib):
    plan, _ = _multi_fns(lib)
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # B=4, 8 query rows, <= 2 per sequence, 8/2 heads, d=128, bs=16, 16 blocks per
    # table, longest context 256, 64-token partitions: 4 partitions per row
    rc, P, W = _multi_plan(plan, 4, 8, 2, 8, 2, 128, 16, 16, 256, 64)
    rows = 8 * 8 * 4
    assert rc == 0 and P == 64 and W == up(rows * 128 * 4) + 2 * up(rows * 4)
    # one partition covers the longest context: no workspace
    rc, P, W = _multi_plan(plan, 4, 8, 2, 8, 2, 128, 16, 16, 64, 64)
    assert rc == 0 and W == 0


@pytest.mark.parametrize("args,status", [
    ((4, 8, 2, 6, 4, 128, 16, 16, 256, 64), -1),    # 6 % 4 != 0
    ((4, 8, 2, 8, 2, 96, 16, 16, 256, 64), -2),     # head_dim 96 not built
    ((4, 8, 2, 8, 2, 128, 8, 16, 256, 64), -2),     # block size not a multiple of 16
    ((4, 8, 2, 6, 2, 128, 16, 16, 256, 64), -2),    # group 3
    ((4, 8, 2, 8, 2, 128, 16, 16, 256, 24), -1),    # partition not a multiple of 16
    ((-1, 8, 2, 8, 2, 128, 16, 16, 256, 64), -1),
    ((4, 8, 2, 8, 2, 128, 16, 0, 256, 64), -1),     # no blocks per table
])
def test_multi_plan_rejects(lib, args, status):
    plan, _ = _multi_fns(lib)
    assert _multi_plan(plan, *args)[0] == status


def test_multi_call_rejects_bad_arguments_without_launching(lib):
    _, att = _multi_fns(lib)
    n = None
    x = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    ws = ctypes.c_void_p(1 << 24)

    def call(out=x, q=x, qs=x, num_blocks=40, scale=0.1, B=4, ws_ptr=ws, ws_bytes=1 << 22,
             max_len=256, P=64):
        return att(out, q, x, x, x, x, qs, B, 8, 2, 16, num_blocks, scale, 8, 2, 128, 16,
                   max_len, P, ws_ptr, ws_bytes, n, n, n)
    assert call(num_blocks=0) == -1
    assert call(scale=float("nan")) == -1
    assert call(out=n) == -1
    assert call(q=odd) == -1
    assert call(qs=n) == -1
    assert call(ws_ptr=n) == -3                       # 4 partitions, no workspace
    assert call(ws_bytes=64) == -3
    assert call(B=0) == 0                             # nothing to do
    assert call(num_blocks=1 << 27) == -2             # TMA rows past 32 bits


def test_prefix_shared_call_rejects_bad_arguments(lib):
    c = ctypes
    p = c.c_void_p
    fn = lib.paged_decode_attention_prefix_shared
    fn.argtypes = [p, p, p, p, p, p, c.c_int, c.c_int, c.c_int64, c.c_float, c.c_int, c.c_int,
                   c.c_int, c.c_int, c.c_int, p, p, c.c_int, c.c_int, c.c_int, p, c.c_size_t, p,
                   p, p]
    fn.restype = c.c_int
    x = p(1 << 20)
    odd = p((1 << 20) + 2)

    def call(num_blocks=40, scale=0.1, offs=x, pref=x, groups=2):
        return fn(x, x, x, x, x, x, 4, 8, num_blocks, scale, 8, 2, 128, 16, 256, offs, pref,
                  groups, 2, 64, x, 1 << 22, None, None, None)
    assert call(num_blocks=0) == -1
    assert call(scale=float("inf")) == -1
    assert call(offs=None) == -1                      # groups without their offsets
    assert call(pref=None) == -1
    assert call(offs=odd) == -1                       # int32 arrays must be 4-byte aligned
    ex = lib.paged_decode_attention_prefix_shared_ex
    ex.argtypes = fn.argtypes + [c.c_uint32]
    ex.restype = c.c_int
    # unknown flag bits are rejected first; the flag itself changes no host check
    assert ex(x, x, x, x, x, x, 4, 8, 40, 0.1, 8, 2, 128, 16, 256, x, x, 2, 2, 64, x, 1 << 22,
              None, None, None, 0x4) == -1
    assert ex(x, x, x, x, x, x, 4, 8, 0, 0.1, 8, 2, 128, 16, 256, x, x, 2, 2, 64, x, 1 << 22,
              None, None, None, pkv.PKV_TABLES_READY) == -1
