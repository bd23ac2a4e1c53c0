"""The C ABI from a plain C program (tests/c/qsa_c_client.c): no Python, no
PyTorch on the call path. On the CPU it checks the host-side contract; on a
GPU it runs one decode on cudaMalloc'd buffers, whose output the oracle checks."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from sparse_attention_paged_qsa_gb300 import binding as B
from sparse_attention_paged_qsa_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "qsa_c_client.c")


def _client(tmp_path):
    libbuild.build_library()
    cuda = os.path.dirname(os.path.dirname(libbuild.nvcc()))
    exe = tmp_path / "qsa_c_client"
    subprocess.run(["gcc", "-O1", "-std=c11", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), SRC, "-o", str(exe),
                    "-L", os.path.dirname(B.LIB_PATH), "-lqsa", "-L", os.path.join(cuda, "lib64"),
                    "-lcudart", "-Wl,-rpath," + os.path.dirname(B.LIB_PATH)],
                   check=True)
    return exe


def test_c_client_host_contract(tmp_path):
    exe = _client(tmp_path)
    r = subprocess.run([str(exe), "host"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("host ok")


@pytest.mark.gpu
def test_c_client_decode_matches_the_oracle(tmp_path):
    exe = _client(tmp_path)
    r = subprocess.run([str(exe), "gpu", str(tmp_path)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    bs, hq, d, slots = 3, 12, 256, 4096
    rd = lambda n, dt: np.fromfile(tmp_path / n, dtype=dt)
    q = rd("q.bin", np.uint16).reshape(bs, hq, d)
    k = rd("k.bin", np.uint16).reshape(slots, 1, d)
    v = rd("v.bin", np.uint16).reshape(slots, 1, d)
    sel, cu = rd("sel.bin", np.int32), rd("cu.bin", np.int32)
    out = rd("out.bin", np.uint16).reshape(bs, hq, d)
    ref = oracle.round_bf16(oracle.decode(q, k, v, "bf16", sel, cu, 1 / 16))
    got = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    num = np.sqrt(((got - ref) ** 2).sum(-1))
    den = np.sqrt((ref ** 2).sum(-1))
    assert (num / den).max() <= 2e-3
