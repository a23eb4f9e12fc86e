"""The C ABI from plain C: paged_kv_cache_213_gb300/examples/decode_step.c
includes include/pagedkv.h, links libpagedkv and runs plan, workspace clear,
decode step and error read on one stream.

Without a GPU the example must compile as strict C99 against the header and
link against the library (every entry it calls is exported).  On a GPU it
runs, and its output is checked against the oracle: the appended step's
attention over the file's own inputs."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import paged_kv_cache_213_gb300 as pkv
from paged_kv_cache_213_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "paged_kv_cache_213_gb300", "examples", "decode_step.c")


def _cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cudart_dir(home):
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(home, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return None


def compile_example(out_path):
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    pkv_build.build()
    home = _cuda_home()
    libdir = _cudart_dir(home)
    if libdir is None:
        pytest.skip("libcudart.so not found")
    libpkv = os.path.dirname(pkv.library_path())
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O2",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(home, "include"),
           SRC, "-L", libpkv, "-lpagedkv", "-L", libdir, "-lcudart", "-lm",
           f"-Wl,-rpath,{libpkv}", f"-Wl,-rpath,{libdir}", "-o", out_path]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out_path


def test_example_compiles_as_c99_and_links(tmp_path):
    exe = compile_example(str(tmp_path / "decode_step"))
    assert os.path.getsize(exe) > 0


def _read(path):
    raw = open(path, "rb").read()
    pos = 0

    def take(dtype, count):
        nonlocal pos
        a = np.frombuffer(raw, dtype=dtype, count=count, offset=pos)
        pos += a.nbytes
        return a

    B, H, HK, D, BS, NB, MB, part, bits = (int(x) for x in take(np.int32, 9))
    f = {"B": B, "H": H, "HK": HK, "D": D, "BS": BS, "NB": NB, "MB": MB, "part": part,
         "bits": bits}
    f["lens"] = take(np.int32, B)
    f["tables"] = take(np.int32, B * MB).reshape(B, MB)
    f["slots"] = take(np.int64, B)
    f["q"] = take(np.float16, B * H * D).reshape(B, H, D)
    f["k_new"] = take(np.float16, B * HK * D).reshape(B, HK, D)
    f["v_new"] = take(np.float16, B * HK * D).reshape(B, HK, D)
    f["k_cache"] = take(np.float16, NB * HK * BS * D).reshape(NB, HK, BS, D)
    f["v_cache"] = take(np.float16, NB * HK * BS * D).reshape(NB, HK, BS, D)
    f["out"] = take(np.float16, B * H * D).reshape(B, H, D)
    f["lse"] = take(np.float32, B * H).reshape(B, H)
    assert pos == len(raw)
    return f


@pytest.mark.gpu
def test_example_runs_and_matches_the_oracle(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    exe = compile_example(str(tmp_path / "decode_step"))
    out_file = str(tmp_path / "step.bin")
    r = subprocess.run([exe, out_file], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    f = _read(out_file)
    assert f["bits"] == 0 and f["part"] == 0  # no device error; the balanced split
    k2, v2 = oracle.append(f["k_new"], f["v_new"], f["slots"], f["k_cache"], f["v_cache"],
                           f["BS"])
    ref, ref_lse, _ = oracle.decode(f["q"], k2, v2, f["tables"], f["lens"],
                                    1.0 / np.sqrt(f["D"]), f["H"], f["HK"], f["D"], f["BS"])
    got = f["out"].astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 2e-3
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2
    assert np.max(np.abs(f["lse"].astype(np.float64) - ref_lse)) <= 1e-4
