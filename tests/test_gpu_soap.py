"""GPU parity of the SOAP mode (okls_config.method = SOAP) against the
float64 oracle, through the C ABI: the one-CTA kernels, the batched path with
the logged-rotation eigensolver (sides up to 544) and with the blocked Jacobi
(past 544, or forced past 128).

Teacher-forced: every step starts the oracle from the GPU's own state
(M, V, L, R, Q_L, Q_R).  Bars: M, V, L, R to 1e-5 (fp32 arithmetic), the step
N to 1e-4 (2e-2 with bf16 parameters, which round the new W); after a refresh
the bases must be orthogonal and diagonalise L, R (1e-5), carry decreasing
eigenvalues and agree in sign with the previous bases (orthogonality to
1e-5 d in Frobenius norm, sqrt(d / 128) of that past d = 128: fp32
rotations and d-deep fp32 sums, whose rounding grows like sqrt(d)), and every eigenvector
whose eigenvalue is separated from its neighbours by more than 1e-3 of the
spectrum must match the oracle's within 2e-6 ||L||_F / gap: twice the
solver's stopping residual (1e-6 of the matrix in Frobenius norm, sqrt(d /
128) of that past d = 128, where the fp32 floor of the rotations grows)
over the gap, the first-order bound on an eigenvector's error.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from kronecker_factored_second_gb300 import _lib as L

pytestmark = pytest.mark.gpu

PARTS = [("M", L.STATE_M), ("L", L.STATE_SA), ("R", L.STATE_SB), ("QL", L.STATE_PA), ("QR", L.STATE_PB),
         ("V", L.STATE_V)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()  # fail loudly when the library is missing
    torch.cuda.set_device(0)


def _batch(B, m, n, **kw):
    from kronecker_factored_second_gb300.okls import OklsBatch
    return OklsBatch(B, m, n, method="soap", **kw)


def _snap(ob):
    torch.cuda.synchronize()
    return {k: ob.get_state(p).double().cpu().numpy() for k, p in PARTS}


def _check_basis(Q, S, Q_prev, Q_ref):
    d = S.shape[0]
    out = {}
    # fp32 rotations: orthogonality holds to ~1e-6 per entry, so the
    # Frobenius norm of Q^T Q - I is held to 1e-5 d
    out["orth"] = float(np.linalg.norm(Q.T @ Q - np.eye(d))) / d
    D = Q.T @ S @ Q
    out["offdiag"] = float(np.linalg.norm(D - np.diag(np.diag(D))) / max(np.linalg.norm(S), 1e-30))
    lam = np.diag(D)
    out["order"] = float(max(0.0, np.max(lam[1:] - lam[:-1]) / max(np.abs(lam).max(), 1e-30))) if d > 1 else 0.0
    out["sign"] = float(max(0.0, -np.min(np.sum(Q * Q_prev, axis=0))))
    # eigenvectors with a clear gap must match the oracle's
    w = np.linalg.eigvalsh(0.5 * (S + S.T))[::-1]
    scale = max(abs(w).max(), 1e-30)
    gaps = np.full(d, np.inf)
    if d > 1:
        gaps[:-1] = np.minimum(gaps[:-1], w[:-1] - w[1:])
        gaps[1:] = np.minimum(gaps[1:], w[:-1] - w[1:])
    sel = gaps > 1e-3 * scale
    err = np.linalg.norm(Q[:, sel] - Q_ref[:, sel], axis=0)
    out["vec"] = float(np.max(err)) if sel.any() else 0.0
    # first-order perturbation: ||dq_j|| <= ||dL|| / gap_j, and the solver
    # stops at an off-diagonal residual of 1e-6 of the matrix in Frobenius
    # norm: the error times the gap over ||L||_F is bounded by that residual
    out["vec_gap"] = float(np.max(err * gaps[sel])) / max(float(np.linalg.norm(S)), 1e-30) if sel.any() else 0.0
    return out


@pytest.mark.parametrize("B,m,n,dtype", [(1, 128, 64, torch.float32), (3, 40, 24, torch.float32),
                                         (2, 17, 33, torch.float32), (2, 64, 32, torch.bfloat16)])
def test_teacher_forced_steps(B, m, n, dtype):
    _teacher_forced(B, m, n, dtype)


# the batched-GEMM path: m or n past 128 (or forced); eigensolves in shared
# memory up to 128, past it by logged rotations (the matrix a packed triangle
# in shared memory up to 330, a full one in L2 past that)
@pytest.mark.parametrize("B,m,n,dtype", [(2, 200, 150, torch.float32), (1, 300, 140, torch.float32),
                                         (2, 96, 64, torch.float32), (1, 160, 340, torch.bfloat16),
                                         (1, 544, 331, torch.float32)])  # the largest side; an odd one past 330
def test_teacher_forced_steps_large_path(B, m, n, dtype, monkeypatch):
    monkeypatch.setenv("OKLS_SOAP_LARGE", "1")
    _teacher_forced(B, m, n, dtype)


# the eigensolver with fewer CTAs per matrix, as larger batches take it: one
# CTA (packed triangle in shared memory for d <= 330, full matrix in L2
# past it) and clusters of 2 over the matrix in L2
@pytest.mark.parametrize("B,m,n,dtype,ctas", [(2, 200, 150, torch.float32, 1), (1, 160, 340, torch.float32, 1),
                                              (1, 160, 340, torch.float32, 2)])
def test_large_path_fewer_ctas_per_matrix(B, m, n, dtype, ctas, monkeypatch):
    monkeypatch.setenv("OKLS_SOAP_LARGE", "1")
    monkeypatch.setenv("OKLS_EIG_CTAS", str(ctas))
    _teacher_forced(B, m, n, dtype)


# the blocked Jacobi refresh (sides past 544; forced past 128 here so that the
# oracle stays quick): padded sides (140 -> 192, 340 -> 384, 600 -> 640), a
# side of 64-multiple size, and one that stays on the one-CTA solver
@pytest.mark.parametrize("B,m,n,dtype,force", [(2, 200, 150, torch.float32, True),
                                               (1, 300, 140, torch.float32, True),
                                               (1, 160, 340, torch.bfloat16, True),
                                               (1, 600, 100, torch.float32, False),
                                               (1, 576, 640, torch.float32, False)])
def test_teacher_forced_steps_blocked_solver(B, m, n, dtype, force, monkeypatch):
    monkeypatch.setenv("OKLS_SOAP_LARGE", "1")
    if force:
        monkeypatch.setenv("OKLS_SOAP_BLOCKED", "1")
    _teacher_forced(B, m, n, dtype)


def _teacher_forced(B, m, n, dtype):
    lr, b1, b2, eps, f = 0.01, 0.9, 0.95, 1e-8, 2
    ob = _batch(B, m, n, param_dtype=dtype, lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, root_every=f)
    rng = np.random.default_rng(m + n)
    W = torch.tensor(rng.standard_normal((B, m, n)) * 0.001, dtype=dtype, device="cuda")
    worst = {}
    for t in range(1, 6):
        pre = _snap(ob)
        Wp = W.double().cpu().numpy()
        G = torch.tensor(rng.standard_normal((B, m, n)), dtype=dtype, device="cuda")
        ob.step(W, G, lr)
        assert ob.query_status() == 0
        post = _snap(ob)
        Wn = W.double().cpu().numpy()
        Gd = G.double().cpu().numpy()
        for b in range(B):
            st = O.SoapState(M=pre["M"][b], V=pre["V"][b], L=pre["L"][b], R=pre["R"][b], QL=pre["QL"][b],
                             QR=pre["QR"][b], t=t - 1)
            ost, _Wo, No = O.soap_step(st, Wp[b], Gd[b], lr, b1, b2, eps, f)
            err = {k: O.rel_fro(post[k][b], getattr(ost, k)) for k in ("M", "V", "L", "R")}
            err["N"] = O.rel_fro((Wp[b] - Wn[b]) / lr, No)
            if t % f == 0:
                for side, S in (("QL", post["L"][b]), ("QR", post["R"][b])):
                    ref = O.eigenvectors_aligned(S, pre[side][b])
                    for k, v in _check_basis(post[side][b], S, pre[side][b], ref).items():
                        err[side + "_" + k] = v
            else:
                err["Q_same"] = float(not (np.array_equal(post["QL"][b], pre["QL"][b])
                                           and np.array_equal(post["QR"][b], pre["QR"][b])))
            for k, v in err.items():
                worst[k] = max(worst.get(k, 0.0), v)
    print(f"soap {B}x{m}x{n} {dtype}", {k: f"{v:.1e}" for k, v in worst.items()})
    for k in ("M", "V", "L", "R"):
        assert worst[k] < 1e-5, (k, worst)
    # bf16 parameters round the new W to 8 bits (|W| ~ 5 lr |N| here): ~1% of the step
    assert worst["N"] < (2e-2 if dtype == torch.bfloat16 else 1e-4), worst
    assert worst["Q_same"] == 0.0
    for side in ("QL", "QR"):
        grow = max(1.0, (m if side == "QL" else n) / 128) ** 0.5
        assert worst[side + "_orth"] < 1e-5 * grow and worst[side + "_offdiag"] < 1e-5, worst
        assert worst[side + "_order"] < 1e-6 and worst[side + "_sign"] == 0.0, worst
        # the solver's stopping residual is 1e-6 up to d = 128, sqrt(d / 128) of that past it
        assert worst[side + "_vec_gap"] < 2e-6 * grow, worst
    ob.close()


@pytest.mark.parametrize("B,m,n,large", [(2, 24, 16, False), (2, 320, 192, True)])
def test_without_refresh_the_step_is_adam(B, m, n, large, monkeypatch):
    """Before any refresh the bases are the identity: SOAP is Adam with both
    moments bias-corrected.  On the batched path (320 x 192) the rotations
    are tensor-core products of three-term bf16 splits: the identity's split
    is exact, so the rotations return G and N' to within fp32 rounding (an
    fp32 value's three terms hold it exactly)."""
    if large:
        monkeypatch.setenv("OKLS_SOAP_LARGE", "1")
    lr, b1, b2, eps = 0.02, 0.9, 0.99, 1e-8
    ob = _batch(B, m, n, lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, root_every=1000)
    rng = np.random.default_rng(3)
    W = torch.zeros((B, m, n), device="cuda")
    Mn = np.zeros((B, m, n))
    Vn = np.zeros((B, m, n))
    Wn = np.zeros((B, m, n))
    for t in range(1, 6):
        G = rng.standard_normal((B, m, n)).astype(np.float32)
        ob.step(W, torch.tensor(G, device="cuda"), lr)
        Mn = b1 * Mn + (1 - b1) * G
        Vn = b2 * Vn + (1 - b2) * G.astype(np.float64) ** 2
        Wn -= lr * (Mn / (1 - b1 ** t)) / (np.sqrt(Vn / (1 - b2 ** t)) + eps)
    assert ob.query_status() == 0
    assert O.rel_fro(W.double().cpu().numpy(), Wn) < 1e-5
    ob.close()


def test_optimizer_class_matches_the_batch_api():
    from kronecker_factored_second_gb300.okls import SOAP, OklsBatch
    torch.manual_seed(5)
    p = torch.nn.Parameter(torch.randn(2, 32, 48, device="cuda") * 0.02)
    W = p.detach().clone()
    opt = SOAP([p], lr=0.01, betas=(0.9, 0.95), eps=1e-8, precondition_frequency=2)
    ob = OklsBatch(2, 32, 48, lr=0.01, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, root_every=2,
                   method="soap")
    for _ in range(4):
        g = torch.randn(2, 32, 48, device="cuda")
        p.grad = g.clone()
        opt.step()
        ob.step(W, g, 0.01)
    torch.cuda.synchronize()
    assert torch.equal(p.detach(), W)
    ob.close()


def _snap_one(ob, b):
    torch.cuda.synchronize()
    return {k: ob.get_state(p)[b].double().cpu().numpy() for k, p in PARTS}


@pytest.mark.parametrize("gi", [0, 1, 2])
def test_full_size_layer_shapes(gi):
    """SOAP on the 1.2B-shaped layer set's shape groups at full size (2048^2,
    5504 x 2048 and 2048 x 5504, bf16 W and G; one layer's batch of each):
    four steps with a refresh every two, so that the first refresh starts
    from the identity and the second from the previous bases.  One matrix per
    group is checked teacher-forced at every step (M, V, L, R, N) and at the
    refreshes its bases (orthogonality, diagonalisation, order, signs and the
    gapped eigenvectors against float64 eigenvectors of the GPU's L, R), with
    the bars of the smaller shapes (sqrt(d / 128) where they grow with d)."""
    from kronecker_factored_second_gb300.okls import OklsBatch
    from kronecker_factored_second_gb300.workloads import GradientStream, workload
    import time

    wl = workload("llama1.2b", layers=1)
    g = wl.groups[gi]
    gs = GradientStream(wl, "cuda")
    lr, b1, b2, eps, f = 0.01, 0.95, 0.95, 1e-8, 2
    ob = OklsBatch(g.batch, g.m, g.n, param_dtype=g.dtype, method="soap", lr=lr, beta1=b1, beta2=b2, eps=eps,
                   weight_decay=0.0, root_every=f)
    W = gs.init_weights(gi)
    b = g.batch - 1
    m, n = g.m, g.n
    worst = {}
    for t in range(1, 5):
        pre = _snap_one(ob, b)
        Wp = W[b].double().cpu().numpy()
        G = gs.grad(gi, t)
        torch.cuda.synchronize()
        t0 = time.time()
        ob.step(W, G, lr)
        assert ob.query_status() == 0
        torch.cuda.synchronize()
        dt = time.time() - t0
        post = _snap_one(ob, b)
        Wn = W[b].double().cpu().numpy()
        Gd = G[b].double().cpu().numpy()
        st = O.SoapState(M=pre["M"], V=pre["V"], L=pre["L"], R=pre["R"], QL=pre["QL"], QR=pre["QR"], t=t - 1)
        # the oracle's own refresh is not needed here: the bases are checked
        # against float64 eigenvectors of the GPU's factors below
        ost, _Wo, No = O.soap_step(st, Wp, Gd, lr, b1, b2, eps, 10 ** 9)
        err = {k: O.rel_fro(post[k], getattr(ost, k)) for k in ("M", "V", "L", "R")}
        err["N"] = O.rel_fro((Wp - Wn) / lr, No)
        if t % f == 0:
            for side, S in (("QL", post["L"]), ("QR", post["R"])):
                ref = O.eigenvectors_aligned(S, pre[side])
                for k, v in _check_basis(post[side], S, pre[side], ref).items():
                    err[side + "_" + k] = v
        print(f"soap {g.name} {m}x{n} t={t} step {dt * 1e3:.0f} ms", {k: f"{v:.1e}" for k, v in err.items()})
        for k, v in err.items():
            worst[k] = max(worst.get(k, 0.0), v)
    ob.close()
    for k in ("M", "V", "L", "R"):
        assert worst[k] < 1e-5, (k, worst)
    # bf16 parameters round the new W to 8 bits
    assert worst["N"] < 2e-2, worst
    for side in ("QL", "QR"):
        grow = max(1.0, (m if side == "QL" else n) / 128) ** 0.5
        assert worst[side + "_orth"] < 1e-5 * grow and worst[side + "_offdiag"] < 1e-5, worst
        assert worst[side + "_order"] < 1e-6 and worst[side + "_sign"] == 0.0, worst
        assert worst[side + "_vec_gap"] < 2e-6 * grow, worst


_CUDA_CORE_SCRIPT = r"""
import os, sys
sys.path.insert(0, os.path.join(os.environ["OKLS_ROOT"], "tests"))
sys.path.insert(0, os.environ["OKLS_ROOT"])
import torch
import test_gpu_soap as T
torch.cuda.set_device(0)
os.environ["OKLS_SOAP_LARGE"] = "1"
os.environ["OKLS_SOAP_BLOCKED"] = "1"
T._teacher_forced(1, 300, 140, torch.float32)   # blocked solver, padded side
os.environ["OKLS_SOAP_BLOCKED"] = "0"
T._teacher_forced(1, 544, 331, torch.float32)   # logged-rotation solver, 544-deep products
"""


def test_cuda_core_products_subprocess():
    """With OKLS_TC3=0 (read once per process, hence a separate one) every
    fp32 product runs on the CUDA cores (k_cl_gemm) and the blocked solver's
    panels on k_bj_rows; the same teacher-forced bars hold there."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, OKLS_TC3="0", OKLS_ROOT=root)
    r = subprocess.run([sys.executable, "-c", _CUDA_CORE_SCRIPT], env=env, timeout=900, capture_output=True, text=True)
    print(r.stdout[-2000:])
    assert r.returncode == 0, r.stderr[-4000:]
