"""A workspace whose arrival counters were not zeroed is flagged instead of
being merged wrong in silence, and paged_decode_workspace_clear recovers it.

The split kernels only count on the per-segment counters (atomic adds) and
never wait on them, and every record address comes from the plan, not from a
count: stale counters change which warp merges (or leave a segment
unmerged), but cannot fault or hang.  A stale value that is negative or at
least the number of pieces counted on it is seen by the first arrival, which
sets PKV_ERRBIT_WORKSPACE; the fills here are of that kind (every byte 0xFF:
counters -1 and NaN records; the bit pattern of 1.0f in every counter).
That arrival also poisons the counter, so a second call on the same stale
workspace is flagged as well, until paged_decode_workspace_clear.  Run on a
batch of few long segments (per-warp kernel) and one of many short segments
(producer/consumer kernel)."""
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


def _batch(which):
    if which == "few":
        return wl.workload(2, poison=True)  # 32 x 8 segments: per-warp ranges
    rng = np.random.default_rng(41)
    return wl.make_batch("many", list(rng.integers(16, 700, size=96)), 32, 8, 128, 16, rng,
                         append=False, poison=True)  # 96 x 8 segments: producer/consumer


def _stale(work, fill):
    if fill == "ff":
        work.fill_(0xFF)
    else:
        work.zero_()
        n = min(work.numel(), pkv.PKV_WORKSPACE_COUNTER_BYTES) // 4
        work[: n * 4].view(torch.float32).fill_(1.0)


@pytest.mark.parametrize("fill", ["ff", "f32_one"])
@pytest.mark.parametrize("which", ["few", "many"])
def test_stale_counters_are_flagged_then_cleared(which, fill):
    batch = _batch(which)
    dev = to_dev(batch)
    if batch.has_append:
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"])
    P, ws = pkv.decode_plan(batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                            batch.block_size, batch.max_blocks_per_seq, batch.max_context_len, 0)
    assert P == 0 and ws > pkv.PKV_WORKSPACE_COUNTER_BYTES
    work = torch.empty(ws, dtype=torch.uint8, device="cuda")
    _stale(work, fill)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        return pkv.paged_decode_attention(
            dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
            batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
            max_context_len=batch.max_context_len, workspace=work, err_word=err)

    call()
    torch.cuda.synchronize()  # returned: stale counts neither fault nor hang
    bits = pkv.get_error(err)
    assert bits == pkv.PKV_ERRBIT_WORKSPACE, bits
    # the flagged counters are poisoned: the next call is flagged again
    err.zero_()
    call()
    assert pkv.get_error(err) == pkv.PKV_ERRBIT_WORKSPACE
    # recovery: clear the counters (the records after them may stay stale)
    pkv.paged_decode_workspace_clear(work)
    err.zero_()
    out = call()
    assert pkv.get_error(err) == 0
    assert_close(out.cpu().numpy(), oracle_step(batch)["out"], what=f"{which} after the clear")
    assert int(work[: pkv.PKV_WORKSPACE_COUNTER_BYTES].view(torch.int32).abs().sum()) == 0


def test_clear_touches_only_the_counter_bytes():
    big = torch.full((2 * pkv.PKV_WORKSPACE_COUNTER_BYTES,), 0xAB, dtype=torch.uint8,
                     device="cuda")
    pkv.paged_decode_workspace_clear(big)
    host = big.cpu().numpy()
    assert not host[: pkv.PKV_WORKSPACE_COUNTER_BYTES].any()
    assert (host[pkv.PKV_WORKSPACE_COUNTER_BYTES:] == 0xAB).all()
    small = torch.full((4096,), 0xAB, dtype=torch.uint8, device="cuda")
    pkv.paged_decode_workspace_clear(small)
    assert not small.cpu().numpy().any()
    pkv.paged_decode_workspace_clear(torch.empty(0, dtype=torch.uint8, device="cuda"))
