"""GPU parity of the Clean mode (okls_config.method = CLEAN; one CTA per
factor for m, n <= 128 and rank + oversample <= 64, batched GEMMs up to
16384 and 544) against the float64 oracle, through the C ABI, up to the
benchmarked layer shapes (2048 and 5504 sides, rank 256 + 8).

Teacher-forced: every step starts the oracle from the GPU's own state.
A refresh step is checked in two parts:
  * the sketch: the oracle's Algorithm 3 on the same Gaussian draws gives
    the reference bases and eigenvalues; the GPU's eigenvalues must match to
    1e-4 max(1, (r + p)/128) of the largest (Jacobi's stopping rule and the
    Gram sums grow with the sketch width), its bases must be orthonormal (1e-5 in Frobenius
    norm over r) and every basis vector whose eigenvalue is separated from
    its neighbours by more than 1e-2 of the largest must match the oracle's
    to 5e-4 (up to sign at the first refresh, where no previous basis fixes
    it): fp32 Gram-Schmidt, Cholesky and Jacobi rotations, whose errors the
    gap divides;
  * the step: the oracle's Algorithm 1 runs on the GPU's new bases (the
    `bases` hook), so the moment transport of Eqns. (14)-(15) and the four
    blocks' moments are compared to 5e-5 (fp32 sums of up to m n terms,
    amplified by the cancellation in the projected blocks) of their norm
    plus an absolute floor at the blocks' rounding scale, e = 4 2^-24
    ||G||_F for a first moment and 2 ||G||_F e for a second one: where the
    sketch is exact (rank + oversample = n here, so both bases are G's
    singular vectors), G_A and G_B vanish and their moments are rounding
    noise on both sides.
The orthogonality bar grows like sqrt(d / 128) past 128 rows of the basis
(fp32 sums over d rows), as SOAP's does.
G~ is checked twice.  Assembly: G~ rebuilt in float64 from the GPU's own
new state (bases, moments, and C = P_L G P_R) must match the applied update
to 1e-5 (2e-2 with bf16 parameters: the new W rounds to 8 bits), plus the
rounding floor of the C term where C itself sits at that floor.  Against the
oracle: G~ is a sum of normalised units (each entry of the Main block, each
column of N(M_A, v_A), each row of N(M_B, v_B), and C), and a unit whose
moment m_u is small against the rounding of the G-linear terms (the e above,
scaled by 1 - beta1 for a first moment) is
ill-conditioned: right after a cold sketch of G G^T the leading columns of
G_A and rows of G_B are the sketch's residual, near that floor, and
normalising them lifts fp32 rounding to a visible share of the unit.  The
error of G~ must stay within the root-sum-square of ||unit|| min(2, base +
e / ||m_u||), base 1e-4 (2e-2 with bf16 parameters).
Between refreshes the bases must stay bit-identical.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from kronecker_factored_second_gb300 import _lib as L

pytestmark = pytest.mark.gpu

PARTS = [("UL", L.STATE_PA), ("UR", L.STATE_PB), ("lamL", L.STATE_SA), ("lamR", L.STATE_SB), ("M", L.STATE_M),
         ("V", L.STATE_V), ("MA", L.STATE_MA), ("MB", L.STATE_MB), ("vA", L.STATE_VA), ("vB", L.STATE_VB),
         ("vC", L.STATE_VC)]
MOMENTS = ("M", "V", "MA", "MB", "vA", "vB", "vC")
MOMENT_BAR = 5e-5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()  # fail loudly when the library is missing
    torch.cuda.set_device(0)


def _batch(B, m, n, **kw):
    from kronecker_factored_second_gb300.okls import OklsBatch
    return OklsBatch(B, m, n, method="clean", **kw)


def _snap(ob):
    torch.cuda.synchronize()
    return {k: ob.get_state(p).double().cpu().numpy() for k, p in PARTS}


def _ostate(pre, b, t):
    cold = t == 0
    return O.CleanState(UL=None if cold else pre["UL"][b], lamL=None if cold else pre["lamL"][b],
                        UR=None if cold else pre["UR"][b], lamR=None if cold else pre["lamR"][b],
                        M=pre["M"][b], V=pre["V"][b], MA=pre["MA"][b], vA=pre["vA"][b], MB=pre["MB"][b],
                        vB=pre["vB"][b], vC=float(pre["vC"][b]), t=t)


def _check_sketch(U, lam, Uo, lamo, aligned):
    """GPU basis U, eigenvalues lam against the oracle's Uo, lamo."""
    r = U.shape[1]
    out = {}
    scale = max(float(np.max(np.abs(lamo))), 1e-30)
    out["lam"] = float(np.max(np.abs(lam - lamo))) / scale
    out["orth"] = float(np.linalg.norm(U.T @ U - np.eye(r))) / r
    s = np.ones(r)
    if not aligned:
        s = np.sign(np.sum(U * Uo, axis=0))
        s[s == 0] = 1.0
    gaps = np.full(r, np.inf)
    if r > 1:
        gaps[:-1] = np.minimum(gaps[:-1], lamo[:-1] - lamo[1:])
        gaps[1:] = np.minimum(gaps[1:], lamo[:-1] - lamo[1:])
    sel = gaps > 1e-2 * scale
    out["vec"] = float(np.max(np.linalg.norm(U[:, sel] * s[sel] - Uo[:, sel], axis=0))) if sel.any() else 0.0
    out["order"] = float(max(0.0, np.max(lam[1:] - lam[:-1]) / scale)) if r > 1 else 0.0
    return out


def _assemble(post, b, G, bc1, bc2, eps):
    """G~ of Eqn. (16) from the GPU's state after the step, in float64, and
    the allowance for its C term: C is recomputed here from G and the GPU's
    bases, so the two differ by the rounding floor e = 4 2^-24 ||G||_F,
    scaled by the GPU's normaliser: negligible unless C itself sits at that
    floor (a basis spanning all of R^n), where the normalised C is noise."""
    UL, UR = post["UL"][b], post["UR"][b]
    PL = np.eye(UL.shape[0]) - UL @ UL.T
    PR = np.eye(UR.shape[0]) - UR @ UR.T
    C = PL @ G @ PR
    main = (post["M"][b] * bc1) / (np.sqrt(post["V"][b] * bc2) + eps)
    bA = (post["MA"][b] * bc1) / (np.sqrt(post["vA"][b] * bc2)[None, :] + eps)
    bB = (post["MB"][b] * bc1) / (np.sqrt(post["vB"][b] * bc2)[:, None] + eps)
    cden = 1.0 / (np.sqrt(post["vC"][b] * bc2) + eps)
    e = 4.0 * 2.0 ** -24 * np.linalg.norm(G)
    allowance = e * cden
    return UL @ main @ UR.T + bA @ UR.T + UL @ bB + C * cden, allowance


def _unit_bound(ost, UL, UR, G, b1, bc1, bc2, eps, base):
    """Root-sum-square over the normalised units of G~ of ||unit|| min(2,
    base + cond), cond = e / ||m_u|| (a normalised unit moves by at most 2
    ||unit||: a sign flip)."""
    m, n = G.shape
    e = 4.0 * 2.0 ** -24 * np.linalg.norm(G)
    tiny = 1e-300
    main = (ost.M * bc1) / (np.sqrt(ost.V * bc2) + eps)
    bA = (ost.MA * bc1) / (np.sqrt(ost.vA * bc2)[None, :] + eps)
    bB = (ost.MB * bc1) / (np.sqrt(ost.vB * bc2)[:, None] + eps)
    PL = np.eye(m) - UL @ UL.T
    PR = np.eye(n) - UR @ UR.T
    C = PL @ G @ PR
    bC = C / (np.sqrt(ost.vC * bc2) + eps)
    terms = [np.abs(main) * np.minimum(2.0, base + (1 - b1) * e / np.maximum(np.abs(ost.M), tiny)),
             np.linalg.norm(bA, axis=0) * np.minimum(2.0, base + (1 - b1) * e /
                                                     np.maximum(np.linalg.norm(ost.MA, axis=0), tiny)),
             np.linalg.norm(bB, axis=1) * np.minimum(2.0, base + (1 - b1) * e /
                                                     np.maximum(np.linalg.norm(ost.MB, axis=1), tiny)),
             np.array([np.linalg.norm(bC) * min(2.0, base + e / max(float(np.linalg.norm(C)), tiny))])]
    return float(np.sqrt(sum(float(np.sum(t * t)) for t in terms)))


def _noise_parts(noise_b, m, p, cold):
    """Psi_L and Psi_R of one matrix as Algorithm 3 takes them: every column
    at the first refresh, the first p beside a previous basis."""
    NL, NR = noise_b[:m], noise_b[m:]
    return (NL, NR) if cold else (NL[:, :p], NR[:, :p])


CASES = [
    # B, m, n, r, p, q, T, dtype, weight_decay, singular values of G
    (2, 96, 64, 8, 4, 1, 2, torch.float32, 0.0, "iid"),
    (2, 96, 64, 8, 4, 1, 2, torch.float32, 0.0, "decay"),
    (1, 128, 128, 32, 16, 1, 2, torch.float32, 0.1, "iid"),
    (3, 40, 24, 6, 2, 0, 1, torch.float32, 0.0, "iid"),
    (2, 17, 33, 4, 3, 2, 3, torch.float32, 0.0, "iid"),
    (2, 48, 16, 12, 4, 1, 2, torch.float32, 0.0, "iid"),   # r + p = n: the right sketch spans R^n
    (2, 64, 32, 8, 8, 1, 2, torch.bfloat16, 0.0, "iid"),
    (2, 20, 12, 1, 0, 1, 2, torch.float32, 0.0, "iid"),      # the smallest basis: r = 1, no oversampling
    (1, 128, 128, 48, 16, 2, 2, torch.float32, 0.0, "iid"),  # the largest sketch: r + p = 64
    (2, 9, 1, 1, 0, 1, 1, torch.float32, 0.0, "iid"),        # n = 1: U_R spans R^1, G_B and C vanish
]

# the batched-GEMM path: m or n past 128, or r + p past 64 (or forced)
LARGE_CASES = [
    (2, 200, 144, 16, 8, 1, 2, torch.float32, 0.0, "iid"),
    (1, 300, 520, 56, 16, 1, 2, torch.float32, 0.1, "iid"),
    (1, 260, 200, 112, 16, 2, 3, torch.float32, 0.0, "decay"),  # the largest sketch: r + p = 128
    (2, 160, 96, 12, 4, 1, 2, torch.bfloat16, 0.0, "iid"),
    (2, 96, 64, 8, 4, 1, 2, torch.float32, 0.0, "iid"),       # a one-CTA shape, forced onto this path
    (2, 260, 180, 131, 6, 1, 2, torch.float32, 0.0, "iid"),   # r + p = 137: packed eigensolve, odd k
    (1, 400, 300, 256, 8, 1, 2, torch.float32, 0.0, "iid"),   # the pages' rank 256 with oversampling 8
    (1, 420, 360, 332, 8, 0, 2, torch.float32, 0.0, "iid"),   # r + p = 340: the eigensolve's matrices in L2
    (1, 600, 560, 536, 8, 0, 2, torch.float32, 0.0, "iid"),   # r + p = 544: the largest sketch
]


@pytest.mark.parametrize("B,m,n,r,p,q,T,dtype,wd,spectrum", CASES)
def test_teacher_forced_steps(B, m, n, r, p, q, T, dtype, wd, spectrum):
    """spectrum "iid": G with iid N(0, 1) factors; "decay": singular values
    1/(1+k), as in a layer's gradient, where the first (cold) sketch is
    nearly exact and its residual blocks are rounding-dominated."""
    _teacher_forced(B, m, n, r, p, q, T, dtype, wd, spectrum)


@pytest.mark.parametrize("B,m,n,r,p,q,T,dtype,wd,spectrum", LARGE_CASES)
def test_teacher_forced_steps_large_path(B, m, n, r, p, q, T, dtype, wd, spectrum, monkeypatch):
    monkeypatch.setenv("OKLS_CLEAN_LARGE", "1")
    _teacher_forced(B, m, n, r, p, q, T, dtype, wd, spectrum)


# the shapes and settings of bench.py's Clean leg on the 1.2B-shaped set
# (rank 256, oversampling 8, one power iteration, bf16 W and G), one matrix
# per shape, a refresh every other step
LAYER_CASES = [
    (1, 2048, 2048, 256, 8, 1, 2, torch.bfloat16, 0.0, "decay"),
    (1, 5504, 2048, 256, 8, 1, 2, torch.bfloat16, 0.0, "decay"),
    (1, 2048, 5504, 256, 8, 1, 2, torch.bfloat16, 0.0, "iid"),
]


@pytest.mark.parametrize("B,m,n,r,p,q,T,dtype,wd,spectrum", LAYER_CASES)
def test_teacher_forced_steps_layer_shapes(B, m, n, r, p, q, T, dtype, wd, spectrum):
    _teacher_forced(B, m, n, r, p, q, T, dtype, wd, spectrum)


def test_rank256_one_cta_per_matrix(monkeypatch):
    """The pages' rank 256 + 8 with the eigensolver on one CTA per matrix
    (the packed-triangle kernel that full layer sets take)."""
    monkeypatch.setenv("OKLS_CLEAN_LARGE", "1")
    monkeypatch.setenv("OKLS_EIG_CTAS", "1")
    _teacher_forced(1, 400, 300, 256, 8, 1, 2, torch.float32, 0.0, "iid")


def _teacher_forced(B, m, n, r, p, q, T, dtype, wd, spectrum):
    lr, b1, b2, eps = 0.01, 0.95, 0.95, 1e-8
    ob = _batch(B, m, n, param_dtype=dtype, lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd, root_every=T,
                rank=r, oversample=p, power_iters=q)
    rng = np.random.default_rng(7 * m + n)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(m * n)
    W = torch.tensor(rng.standard_normal((B, m, n)) * 0.001, dtype=dtype, device="cuda")
    decay = 1.0 - lr * wd
    worst = {}
    for t in range(1, 6):
        pre = _snap(ob)
        due = ob.refresh_due
        assert due == ((t - 1) % T == 0)
        noise = torch.randn(ob.noise_shape, generator=gen, device="cuda") if due else None
        Wp = W.double().cpu().numpy()
        # G = A diag(s) B^T with Gaussian A, B
        s = 1.0 / (1.0 + np.arange(min(m, n))) if spectrum == "decay" else np.ones(min(m, n))
        G = np.einsum("bik,k,bjk->bij", rng.standard_normal((B, m, min(m, n))), s,
                      rng.standard_normal((B, n, min(m, n))))
        Gt = torch.tensor(G, dtype=dtype, device="cuda")
        ob.step(W, Gt, lr, noise=noise)
        assert ob.query_status() == 0
        post = _snap(ob)
        Wn = W.double().cpu().numpy()
        Gd = Gt.double().cpu().numpy()
        nz = noise.double().cpu().numpy() if due else None
        for b in range(B):
            err = {}
            cold = t == 1
            psiL = psiR = None
            if due:
                psiL, psiR = _noise_parts(nz[b], m, p, cold)

                def aL(X, U=None if cold else pre["UL"][b], lm=None if cold else pre["lamL"][b], Gb=Gd[b]):
                    out = (1.0 - b2) * (Gb @ (Gb.T @ X))
                    return out + b2 * (U @ (lm[:, None] * (U.T @ X))) if U is not None else out

                def aR(X, U=None if cold else pre["UR"][b], lm=None if cold else pre["lamR"][b], Gb=Gd[b]):
                    out = (1.0 - b2) * (Gb.T @ (Gb @ X))
                    return out + b2 * (U @ (lm[:, None] * (U.T @ X))) if U is not None else out
                ULo, lamLo = O.nystrom_warm(aL, r, p, q, None if cold else pre["UL"][b], psiL)
                URo, lamRo = O.nystrom_warm(aR, r, p, q, None if cold else pre["UR"][b], psiR)
                for side, U, lam, Uo, lamo in (("L", post["UL"][b], post["lamL"][b], ULo, lamLo),
                                               ("R", post["UR"][b], post["lamR"][b], URo, lamRo)):
                    for k, v in _check_sketch(U, lam, Uo, lamo, aligned=not cold).items():
                        err[side + "_" + k] = v
                bases = (post["UL"][b], post["lamL"][b], post["UR"][b], post["lamR"][b])
            else:
                err["U_same"] = float(not (np.array_equal(post["UL"][b], pre["UL"][b])
                                           and np.array_equal(post["UR"][b], pre["UR"][b])
                                           and np.array_equal(post["lamL"][b], pre["lamL"][b])))
                bases = None
            ost, _Wo, Gto = O.clean_step(_ostate(pre, b, t - 1), Wp[b], Gd[b], lr, b1, b2, eps, r, p, q, T,
                                         psiL, psiR, bases=bases)
            e = 4.0 * 2.0 ** -24 * np.linalg.norm(Gd[b])
            for k in MOMENTS:
                ref = np.asarray(getattr(ost, k), dtype=np.float64)
                floor = e if k in ("M", "MA", "MB") else 2.0 * np.linalg.norm(Gd[b]) * e
                err[k] = float(np.linalg.norm(post[k][b] - ref)) / (float(np.linalg.norm(ref)) + floor / MOMENT_BAR)
            Ng = (decay * Wp[b] - Wn[b]) / lr
            bc1, bc2 = 1.0 / (1.0 - b1 ** t), 1.0 / (1.0 - b2 ** t)
            err["N"] = O.rel_fro(Ng, Gto)  # reported only: see the module docstring
            Gasm, allow = _assemble(post, b, Gd[b], bc1, bc2, eps)
            asm_bar = 2e-2 if dtype == torch.bfloat16 else 1e-5
            # as a fraction of the bar: <= 1 passes
            err["N_asm"] = float(np.linalg.norm(Ng - Gasm)) / (asm_bar * float(np.linalg.norm(Gasm)) + allow)
            bound = _unit_bound(ost, post["UL"][b], post["UR"][b], Gd[b], b1, bc1, bc2, eps,
                                2e-2 if dtype == torch.bfloat16 else 1e-4)
            err["N_units"] = float(np.linalg.norm(Ng - Gto)) / bound
            for k, v in err.items():
                worst[k] = max(worst.get(k, 0.0), v)
    print(f"clean {B}x{m}x{n} r{r} p{p} q{q} T{T} {dtype} {spectrum}", {k: f"{v:.1e}" for k, v in worst.items()})
    for k in MOMENTS:
        assert worst[k] < MOMENT_BAR, (k, worst)
    assert worst["N_asm"] <= 1.0, worst
    assert worst["N_units"] <= 1.0, worst
    assert worst.get("U_same", 0.0) == 0.0
    for side, d in (("L", m), ("R", n)):
        # past k = 128 the k x k stopping rule and Gram sums add error that
        # grows with k; the entries of U^T U are fp32 sums over the basis's d
        # rows, whose rounding grows like sqrt(d) 2^-24 (the bar SOAP's bases
        # take for the same reason: 1e-5, x sqrt(d / 128) past 128 rows)
        orth_bar = 1e-5 * max(1.0, (d / 128) ** 0.5)
        assert worst[side + "_lam"] < 1e-4 * max(1.0, (r + p) / 128) and worst[side + "_orth"] < orth_bar, worst
        assert worst[side + "_order"] == 0.0, worst
        assert worst[side + "_vec"] < 5e-4, worst
    ob.close()


def test_refresh_step_requires_noise():
    ob = _batch(1, 32, 24, rank=4, oversample=2, power_iters=1, root_every=2)
    W = torch.zeros((1, 32, 24), device="cuda")
    G = torch.randn((1, 32, 24), device="cuda")
    with pytest.raises(L.OklsError) as ei:
        ob.step(W, G, 0.01)
    assert ei.value.code == L.OKLS_ERR_INVALID_ARG
    assert ob.t == 0
    ob.step(W, G, 0.01, noise=torch.randn(ob.noise_shape, device="cuda"))
    ob.step(W, G, 0.01)  # t = 2: no refresh, no noise needed
    assert ob.t == 2 and ob.query_status() == 0
    ob.close()


def test_nonfinite_gradient_leaves_w_and_state():
    ob = _batch(2, 32, 24, rank=4, oversample=2, power_iters=1, root_every=3)
    W = torch.randn((2, 32, 24), device="cuda") * 0.01
    ob.step(W, torch.randn((2, 32, 24), device="cuda"), 0.01, noise=torch.randn(ob.noise_shape, device="cuda"))
    assert ob.query_status() == 0
    pre = _snap(ob)
    W0 = W.clone()
    G = torch.randn((2, 32, 24), device="cuda")
    G[1, 3, 5] = float("nan")
    ob.step(W, G, 0.01)
    code, word = ob.status_nothrow()
    assert code == L.OKLS_ERR_NONFINITE and word & L.DEV_NONFINITE_INPUT
    post = _snap(ob)
    assert torch.equal(W[1], W0[1])
    for k in ("UL", "UR", "lamL", "lamR"):
        assert np.array_equal(pre[k], post[k]), k
    ob.close()


def test_optimizer_class_matches_the_batch_api():
    from kronecker_factored_second_gb300.okls import Clean, OklsBatch
    torch.manual_seed(5)
    p = torch.nn.Parameter(torch.randn(2, 48, 40, device="cuda") * 0.02)
    W = p.detach().clone()
    opt = Clean([p], lr=0.01, betas=(0.95, 0.95), eps=1e-8, rank=8, oversample=4, power_iters=1,
                precondition_frequency=2, seed=11)
    ob = OklsBatch(2, 48, 40, lr=0.01, beta1=0.95, beta2=0.95, eps=1e-8, weight_decay=0.0, root_every=2,
                   method="clean", rank=8, oversample=4, power_iters=1)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    for _ in range(5):
        g = torch.randn(2, 48, 40, device="cuda")
        p.grad = g.clone()
        opt.step()
        noise = torch.randn(ob.noise_shape, generator=gen, device="cuda") if ob.refresh_due else None
        ob.step(W, g, 0.01, noise=noise)
    torch.cuda.synchronize()
    assert torch.equal(p.detach(), W)
    ob.close()


def test_cholesky_breakdown_flags_and_leaves_w_and_state():
    """All-zero Gaussian draws at the first refresh make the sketch, and so
    Omega^T Y_nu, zero: the Cholesky factorisation breaks down, the status
    word carries the iteration bit, and neither W nor the state moves."""
    ob = _batch(2, 32, 24, rank=4, oversample=2, power_iters=1, root_every=3)
    W = torch.randn((2, 32, 24), device="cuda") * 0.01
    W0 = W.clone()
    pre = _snap(ob)
    ob.step(W, torch.randn((2, 32, 24), device="cuda"), 0.01, noise=torch.zeros(ob.noise_shape, device="cuda"))
    code, word = ob.status_nothrow()
    assert code == L.OKLS_ERR_NONFINITE and word & L.DEV_NONFINITE_ITER
    assert torch.equal(W, W0)
    post = _snap(ob)
    for k in pre:
        assert np.array_equal(pre[k], post[k]), k
    ob.close()
