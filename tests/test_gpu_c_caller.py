"""The merge's C ABI called from C: tests/c/merge_from_c.c, compiled with gcc
against include/dcp_lse_reduce.h and linked to the library, runs one merge
on cudaMalloc'd buffers with no Python in the call path. Its outputs are
compared with the oracle at the merge's tolerances, and the host-side
rejection of a bad argument (cp = 0) is checked from C too."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import decode_context_mla_dcp_gb300 as dcp
from decode_context_mla_dcp_gb300 import build as dcp_build
from decode_context_mla_dcp_gb300.inputs import make_merge_inputs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(dcp_build.nvcc_path())))


@pytest.fixture(scope="module")
def c_caller(tmp_path_factory):
    gcc = shutil.which("gcc")
    assert gcc is not None, "gcc is needed to build the C caller"
    lib = dcp_build.build()
    lib_dir = os.path.dirname(lib)
    cuda = cuda_home()
    exe = str(tmp_path_factory.mktemp("c_caller") / "merge_from_c")
    cmd = [gcc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c", "merge_from_c.c"),
           "-L", lib_dir, "-ldcp_lse_reduce", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe]
    subprocess.run(cmd, check=True)
    return exe


@pytest.mark.parametrize("cfg,rows,pad", [("kimi", 8, 3), ("deepseek", 5, 0), ("spec", 12, 1)])
def test_merge_called_from_c_matches_the_oracle(oracle_mod, c_caller, tmp_path, cfg, rows, pad):
    inp = make_merge_inputs(cfg, rows, seed=5)
    cp, B, H, D = inp.cp, inp.B, inp.H, inp.D
    stride = H + pad  # padded LSE rows; the padding holds NaN and must never be read
    with open(tmp_path / "in.bin", "wb") as f:
        np.array([cp, H, D, int(inp.lse_base_e)], dtype=np.int32).tofile(f)
        np.array([B, stride], dtype=np.int64).tofile(f)
        for s in inp.srcs:
            np.ascontiguousarray(s, dtype=np.uint16).tofile(f)
        for l in inp.lses:
            padded = np.full((B, stride), np.nan, dtype=np.float32)
            padded[:, :H] = np.asarray(l, dtype=np.float32).reshape(B, H)
            padded.tofile(f)
    run = subprocess.run([c_caller, str(tmp_path / "in.bin"), str(tmp_path / "out.bin")], capture_output=True,
                         text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert f"cp=0 -> {-2}: " in run.stdout and dcp.dcp_lse_reduce_strerror(-2) in run.stdout
    assert f"version {dcp.dcp_lse_reduce_version()}" in run.stdout

    Hl = H // cp
    raw = np.fromfile(tmp_path / "out.bin", dtype=np.uint8)
    n_dst, n_lse = B * Hl * D * 2, B * Hl * 4
    assert raw.size == cp * (n_dst + n_lse)
    ref, lref = oracle_mod.merge(inp.srcs, [np.asarray(l).reshape(B, H) for l in inp.lses], inp.lse_base_e)
    for r in range(cp):
        bits = raw[r * n_dst:(r + 1) * n_dst].view(np.uint16).reshape(B, Hl, D)
        got = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert not np.isnan(got).any()
        err = np.abs(got - ref[r])
        assert (err <= 1e-2 + 8e-3 * np.abs(ref[r])).all(), f"dest {r}: max err {err.max():.3g}"
        lse = raw[cp * n_dst + r * n_lse: cp * n_dst + (r + 1) * n_lse].view(np.float32).reshape(B, Hl)
        lse = lse.astype(np.float64)
        fin = np.isfinite(lref[r])
        assert np.array_equal(np.isfinite(lse), fin)
        assert (np.abs(lse[fin] - lref[r][fin]) <= 1e-5 * np.maximum(np.abs(lref[r][fin]), 1.0)).all()
