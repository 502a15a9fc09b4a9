"""The C ABI from a plain C program: tests/c_abi/okls_c_client.c is compiled
against include/okls.h and libokls.so (no Python in the loop), runs a few
steps with gradients read from a file, and must leave W bit-identical to the
Python binding's run of the same steps on the same library."""

from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from kronecker_factored_second_gb300 import _lib as L

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    pytest.skip("CUDA toolkit headers not found")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    out = str(tmp_path_factory.mktemp("cabi") / "okls_c_client")
    libdir = os.path.dirname(L.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Werror", "-o", out,
                    os.path.join(ROOT, "tests", "c_abi", "okls_c_client.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", libdir, "-lokls", "-Wl,-rpath," + libdir,
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")],
                   check=True, capture_output=True, text=True)
    return out


@pytest.mark.parametrize("method,B,m,n", [(L.METHOD_OKLS, 2, 96, 64), (L.METHOD_SHAMPOO, 1, 64, 40),
                                          (L.METHOD_SOAP, 2, 48, 32)])
def test_c_client_matches_the_python_binding(client, tmp_path, method, B, m, n):
    from kronecker_factored_second_gb300.okls import OklsBatch
    steps = 3
    rng = np.random.default_rng(100 + method)
    G = rng.standard_normal((steps, B, m, n)).astype(np.float32)
    gpath, wpath = tmp_path / "G.bin", tmp_path / "W.out"
    G.tofile(gpath)
    r = subprocess.run([client, str(method), str(B), str(m), str(n), str(steps), str(gpath), str(wpath)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    Wc = np.fromfile(wpath, dtype=np.float32).reshape(B, m, n)

    name = {L.METHOD_OKLS: "okls", L.METHOD_SHAMPOO: "shampoo", L.METHOD_SOAP: "soap"}[method]
    cfg = L.config_default(B, m, n)
    kw = {}
    if method == L.METHOD_SOAP:
        kw = dict(beta1=0.95, beta2=0.95, eps=1e-8, weight_decay=0.0, root_every=2)
    ob = OklsBatch(B, m, n, lr=cfg.lr_peak, method=name, **kw)
    W = torch.zeros((B, m, n), device="cuda")
    for t in range(steps):
        ob.step(W, torch.tensor(G[t], device="cuda"), cfg.lr_peak)
    assert ob.query_status() == 0
    Wp = W.cpu().numpy()
    ob.close()
    assert np.array_equal(Wc, Wp), float(np.max(np.abs(Wc - Wp)))
    assert np.isfinite(Wc).all() and np.abs(Wc).max() > 0
