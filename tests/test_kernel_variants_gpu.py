"""Every decode kernel stays correct on every shape: the CUDA-core kernel
(the only one for block sizes below 16), the tensor-core grid kernel, and the
balanced split on per-warp ranges or on the producer/consumer kernel are each
forced with PKV_DECODE_KERNEL in a child process and checked against the
oracle, also on the shapes where the automatic choice picks another one."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import numpy as np
from gpu_util import assert_close, gpu_step, oracle_step
from paged_kv_cache_213_gb300 import workloads as wl
for cfg in (1, 2, 3):
    batch = wl.workload(cfg, poison=True)
    for P in (0, 64):
        g = gpu_step(batch, partition_tokens=P)
        assert g["err"] == 0
        ref = oracle_step(batch)
        assert_close(g["out"], ref["out"], what=f"{{cfg}} P={{P}}")
import os
balanced = os.environ.get("PKV_DECODE_KERNEL") in ("warp", "pipe")
rng = np.random.default_rng(77)
for d in (64, 128):
    for G in (1, 2, 4, 8):
        batch = wl.make_batch("v", [1, 16, 17, 200, 513], 2 * G, 2, d, 32, rng, append=True,
                              poison=True)
        for P in ((0, 64) if balanced else (64,)):
            g = gpu_step(batch, partition_tokens=P)
            assert g["err"] == 0
            assert_close(g["out"], oracle_step(batch)["out"], what=f"d={{d}} G={{G}} P={{P}}")
if balanced:
    # the balanced split on every KV-head count it takes, ragged and empty sequences
    for Hk in (1, 4, 8, 16):
        for d in (64, 128):
            lens = [0, 1, 15, 16, 17, 100, 700, 33, 2100, 64]
            batch = wl.make_batch("h", lens, 4 * Hk, Hk, d, 16, rng, append=False, poison=True)
            g = gpu_step(batch)
            assert g["err"] == 0
            ref = oracle_step(batch)
            assert_close(g["out"], ref["out"], what=f"Hk={{Hk}} d={{d}}")
            assert np.max(np.abs(g["lse"][1:] - ref["lse"][1:])) <= 1e-4
            assert np.all(np.isneginf(g["lse"][0])) and not np.any(g["out"][0])
if os.environ.get("PKV_DECODE_KERNEL") == "simt":
    from gpu_util import relayout
    base = wl.make_batch("inv", [70, 16, 530, 33], 16, 4, 128, 16, rng, append=False,
                         poison=True)
    out0 = gpu_step(base, partition_tokens=64)["out"]
    for bs, seed in ((1, 5), (8, 6), (32, 7)):
        out = gpu_step(relayout(base, bs, seed), partition_tokens=64)["out"]
        assert np.array_equal(out.view(np.uint16), out0.view(np.uint16)), bs
print("ok")
"""


@pytest.mark.parametrize("kernel", ["simt", "mma", "warp", "pipe"])
def test_forced_kernel(kernel):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tests = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PKV_DECODE_KERNEL=kernel)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, tests=tests)], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
