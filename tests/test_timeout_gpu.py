"""The bounded-wait timeout path, run on purpose without a fault.

Every wait of the decode kernels is bounded (about a second); when one gives
up the kernel flags PKV_ERRBIT_TIMEOUT, waits (bounded) for the copies it has
in flight and stops, so the CUDA context stays usable.  The test hook
PKV_TEST_WAIT_POLLS=0 makes each warp's first wait for K/V data give up at
once, while those copies are still in flight.  The call must return, the
stream must synchronise, the error word must carry the timeout bit, and after
the documented recovery (zero the workspace again) a normal call must match
the oracle.  Run on a batch of few long segments (per-warp kernel) and one of
many short segments (producer/consumer kernel)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_213_gb300 as pkv
from gpu_util import assert_close, oracle_step, to_dev
from paged_kv_cache_213_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _batches():
    rng = np.random.default_rng(41)
    few = wl.workload(2, poison=True)  # 32 x 8 segments: per-warp ranges
    many = wl.make_batch("many", list(rng.integers(16, 700, size=96)), 32, 8, 128, 16, rng,
                         append=False, poison=True)  # 96 x 8 segments: producer/consumer
    return [few, many]


@pytest.mark.parametrize("which", [0, 1])
def test_first_wait_times_out_cleanly_then_recovers(which, monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    batch = _batches()[which]
    dev = to_dev(batch)
    if batch.has_append:
        pkv.paged_kv_append(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"])
    _, ws = pkv.decode_plan(batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                            batch.block_size, batch.max_blocks_per_seq, batch.max_context_len, 0)
    work = torch.zeros(ws, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        return pkv.paged_decode_attention(
            dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
            batch.scale, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
            max_context_len=batch.max_context_len, workspace=work, err_word=err)

    monkeypatch.setenv("PKV_TEST_WAIT_POLLS", "0")
    call()
    torch.cuda.synchronize()  # the kernel returned: no hang, the context is usable
    bits = pkv.get_error(err)
    assert bits & pkv.PKV_ERRBIT_TIMEOUT, bits
    assert not bits & ~pkv.PKV_ERRBIT_TIMEOUT, bits  # no other error on the way
    monkeypatch.delenv("PKV_TEST_WAIT_POLLS")
    # recovery: the arrival counters may be left counted; zero the workspace
    work.zero_()
    err.zero_()
    out = call()
    assert pkv.get_error(err) == 0
    assert_close(out.cpu().numpy(), oracle_step(batch)["out"], what="after the timeout")
    assert float(torch.ones(4, device="cuda").sum()) == 4.0
