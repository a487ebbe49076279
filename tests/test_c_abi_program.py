"""The C ABI from a plain C99 program (tests/c_abi_caller.c): the public header
compiles as C, the program links against libgqa_decode.so with gcc, and its
calls behave as through the Python binding -- host-only calls here, a decode
step on a stream of the program's own against the oracle on the GPU."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import grouped_query_decode_gb300 as gq
import oracle
from gpu_helpers import compare, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cuda_lib_dir():
    for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        p = os.path.join(CUDA, d)
        if os.path.exists(os.path.join(p, "libcudart.so")):
            return p
    pytest.skip("no libcudart.so under CUDA_HOME")


@pytest.fixture(scope="module")
def caller(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib_dir = os.path.dirname(gq.LIB_PATH)
    cuda_lib = _cuda_lib_dir()
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_caller")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(HERE, "c_abi_caller.c"), "-o", exe,
           "-L", lib_dir, "-l:" + os.path.basename(gq.LIB_PATH), "-L", cuda_lib, "-lcudart",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_host_calls(caller):
    r = subprocess.run([caller, "plan"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert int(got["plan_status"]) == gq.GQA_OK
    assert int(got["plan_row_tiles"]) == 1 and int(got["plan_tile_tokens"]) == 64
    assert int(got["plan_max_tiles"]) == 16 * 8 * (4096 // 64)
    assert int(got["head_ratio"]) == gq.GQA_ERR_HEAD_RATIO
    assert int(got["bad_head_dim"]) == gq.GQA_ERR_UNSUPPORTED
    assert int(got["null_pointers"]) == gq.GQA_ERR_INVALID_ARG
    assert got["strerror_ok"] == "yes"


@pytest.mark.gpu
@pytest.mark.parametrize("H,G,sq", [(16, 4, 2), (32, 1, 1)], ids=["gqa-sq2", "mqa"])
def test_c_program_decode_step_vs_oracle(caller, tmp_path, H, G, sq):
    B, D, Tmax = 3, 128, 300
    q, k, v, lens = make_inputs(B, sq, H, G, D, Tmax, [300, 129, 0], seed=1601 + H)
    scale = 1 / math.sqrt(D)
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([B, sq, H, G, D, Tmax], dtype=np.int32).tobytes())
        f.write(np.array([scale], dtype=np.float32).tobytes())
        for a in (q, k, v):
            f.write(np.ascontiguousarray(a, dtype=np.uint16).tobytes())
        f.write(np.ascontiguousarray(lens, dtype=np.int32).tobytes())
    r = subprocess.run([caller, "run", str(inp), str(outp)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    raw = outp.read_bytes()
    nq = B * sq * H * D
    out_bits = np.frombuffer(raw[:2 * nq], dtype=np.uint16).reshape(B, sq, H, D)
    lse = np.frombuffer(raw[2 * nq:], dtype=np.float32).reshape(B, sq, H).astype(np.float64)
    out = (out_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref_out, ref_lse = oracle.gqa_decode_f64(q, k, v, lens, scale, threads=8)
    compare(out, lse, ref_out, ref_lse, what=f"C caller H={H} G={G} sq={sq}")
