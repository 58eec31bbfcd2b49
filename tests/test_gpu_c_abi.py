"""The C ABI without Python: tests/c_abi_consumer.c, compiled with gcc
against include/specverify.h and the CUDA runtime alone, runs the chain and
tree verifies on its own stream; its outputs must equal the oracle's and the
Python binding's."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_36_gb300 as sv
from speculative_decoding_verification_36_gb300 import _lib
from speculative_decoding_verification_36_gb300 import workloads as wl
from parity import chain_report

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _build_consumer(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(_lib.LIB_PATH)
    exe = str(tmp_path / "c_abi_consumer")
    cmd = [cc, "-O2", "-std=c99", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(HERE, "c_abi_consumer.c"), "-o", exe,
           "-L", libdir, "-l:libspecverify.so", f"-Wl,-rpath,{libdir}",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_consumer_matches_oracle_and_binding(tmp_path):
    _lib.load()  # the library is built
    exe = _build_consumer(tmp_path)
    p = wl.preset("c3", B=6, K=4, V=4096)
    x = wl.make_chain(p, seed=13)
    tp = wl.preset("c5", B=6, depth=3, V=4096)
    tr = wl.make_tree(tp, seed=13)
    B, K, V, N = p.B, p.K, p.V, tr["tokens"].shape[1]
    seed = 77
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([B, K, V, N], dtype=np.int32).tobytes())
        f.write(np.array([p.temperature], dtype=np.float32).tobytes())
        f.write(np.array([seed], dtype=np.uint64).tobytes())
        for t in (x["target"], x["draft"]):
            f.write(t.view(torch.int16).numpy().tobytes())
        f.write(x["tokens"].numpy().tobytes())
        f.write(tr["target"].view(torch.int16).numpy().tobytes())
        f.write(tr["tokens"].numpy().tobytes())
        f.write(tr["parents"].numpy().tobytes())
    res = subprocess.run([exe, str(inp), str(out)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    raw = np.fromfile(out, dtype=np.int32)
    W = (N + 31) // 32
    sizes = [B * (K + 1), B, B * (N + 1), B, B * N * W, 1]
    parts = np.split(raw, np.cumsum(sizes)[:-1])
    tokens, n = parts[0].reshape(B, K + 1), parts[1]
    path, length, mask = parts[2].reshape(B, N + 1), parts[3], parts[4].reshape(B, N, W).view(np.uint32)
    assert int(parts[5][0]) == 0  # status flags
    # the oracle
    ref = oracle.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, seed)
    assert not chain_report(tokens, n, ref)["mismatch"]
    tref = oracle.tree_verify_greedy(tr["target"], tr["tokens"], tr["parents"])
    assert np.array_equal(path, tref["path"]) and np.array_equal(length, tref["length"])
    assert np.array_equal(mask, tref["mask"])
    # the Python binding on the same inputs
    dev = torch.device("cuda", 0)
    tb, nb = sv.spec_verify(x["target"].to(dev), x["draft"].to(dev), x["tokens"].to(dev), p.temperature, seed)
    torch.cuda.synchronize()
    assert np.array_equal(tb.cpu().numpy(), tokens) and np.array_equal(nb.cpu().numpy(), n)
