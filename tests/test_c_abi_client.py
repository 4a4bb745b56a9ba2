"""The C ABI from plain C: tests/c_abi/abi_client.c includes only
include/dualkv.h and the CUDA runtime.  On CPU it must compile and link
against libdualkv.so as C99 (the header is valid C).  On the GPU its
outputs must equal, bit for bit, the Python binding's on the same inputs
(deterministic reduction mode)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_client.c")
PKG = os.path.join(ROOT, "shared_prompt_exact_dualkv_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    from shared_prompt_exact_dualkv_gb300 import build
    if not os.path.exists(build.LIB_PATH):
        build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "abi_client")
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Werror", SRC, "-o", exe, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", PKG, "-ldualkv", "-L", os.path.join(CUDA, "lib64"),
           "-lcudart", f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_client_compiles_as_c99(tmp_path):
    assert os.path.exists(_compile(str(tmp_path)))


def _read(d, name, dtype, shape):
    a = np.fromfile(os.path.join(d, name + ".bin"), dtype=dtype).reshape(shape)
    return torch.from_numpy(a.copy())


@pytest.mark.gpu
def test_client_matches_python_binding(tmp_path):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    P, R, Hq, Hkv, d = 200, (150, 0, 131), 4, 2, 128
    T = P + sum(R)
    bf = lambda name, H: _read(tmp_path, name, np.int16, (T, H, d)).view(torch.bfloat16)
    q, k, v, do = bf("q", Hq).cuda(), bf("k", Hkv).cuda(), bf("v", Hkv).cuda(), bf("dout", Hq).cuda()
    scale = np.float32(1.0 / np.sqrt(128.0))
    out, lse = D.forward(q, k, v, P, R, float(scale))
    dq, dk, dv = D.backward(q, k, v, out, do, lse, P, R, float(scale), deterministic=True, num_splits=2)
    assert torch.equal(out.cpu(), bf("out", Hq))
    assert torch.equal(lse.cpu(), _read(tmp_path, "lse", np.float32, (Hq, T)))
    assert torch.equal(dq.cpu(), bf("dq", Hq))
    assert torch.equal(dk.cpu(), bf("dk", Hkv))
    assert torch.equal(dv.cpu(), bf("dv", Hkv))
