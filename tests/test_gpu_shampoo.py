"""GPU parity of the classic Shampoo mode (okls_config.method = SHAMPOO)
against the float64 oracle, through the C ABI.

The step (optim-book "Shampoo" chapter): L += G G^T, R += G^T G,
W -= lr L^-1/4 G R^-1/4, the quarter roots by two chained Newton-Schulz
runs.  Bars: the page's hand example to its printed values within the
ridge's shift; teacher-forced whole steps with L, R to 1e-3, P to 1e-2
against the exact quarter root of the GPU's own ridged factor and to 3e-3
against the chained binary16 replay, U to 2e-2 against the oracle's float64
step and to 1e-2 against the whitening with the GPU's own roots.

Also here: a Newton-Schulz chain that fails (OKLS mode, no ridge, a
rank-deficient factor) leaves the previous roots and their scales together,
so the next step still whitens with them.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import hyper_of, snapshot, spd
from kronecker_factored_second_gb300 import _lib as L

pytestmark = pytest.mark.gpu

HAND_G = [[3.0, 0.0, 1.0], [1.0, 2.0, 0.0]]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()  # fail loudly when the library is missing
    torch.cuda.set_device(0)


def _batch(B, m, n, **kw):
    from kronecker_factored_second_gb300.okls import OklsBatch
    return OklsBatch(B, m, n, method="shampoo", **kw)


def _sv(X):
    return np.sort(np.linalg.svd(X, compute_uv=False))[::-1]


@pytest.mark.parametrize("split,ridge", [(0, 1e-3), (3, 1e-4)])
def test_hand_example_through_the_step(split, ridge):
    """The page's 2 x 3 gradient fed 100 times: the steps at t = 1, 4, 100
    have singular values 1, 0.5, 0.1 (printed to 1e-3); 10 G gives the same
    first step.  The ridge moves them by up to rho ||L||_F / (4 lambda_min)
    (1.7e-3 at rho = 1e-3) and binary16 by ~1e-3: bar 2.5e-3 relative."""
    ob = _batch(1, 2, 3, eps=1e-9, weight_decay=0.0, ridge=ridge, ns_split_iters=split)
    G = torch.tensor([HAND_G], dtype=torch.float32, device="cuda")
    W = torch.zeros_like(G)
    got = {}
    for t in range(1, 101):
        prev = W.clone()
        ob.step(W, G, 1.0)
        if t in (1, 4, 100):
            assert ob.query_status() == 0
            got[t] = _sv((prev - W)[0].double().cpu().numpy())
    for t, want in [(1, 1.0), (4, 0.5), (100, 0.1)]:
        assert np.allclose(got[t], [want, want], rtol=2.5e-3), (t, got[t])
    ob10 = _batch(1, 2, 3, eps=1e-9, weight_decay=0.0, ridge=ridge, ns_split_iters=split)
    W10 = torch.zeros_like(G)
    ob10.step(W10, 10.0 * G, 1.0)
    assert ob10.query_status() == 0
    assert np.allclose(_sv(-W10[0].double().cpu().numpy()), [1.0, 1.0], rtol=2.5e-3)
    ob.close()
    ob10.close()


def _kron_grads(B, m, n, steps, seed, cond=100.0):
    rng = np.random.default_rng(seed)
    out = []
    A = [np.linalg.cholesky(spd(m, cond, seed * 100 + b)) for b in range(B)]
    C = [np.linalg.cholesky(spd(n, cond, seed * 100 + 50 + b)) for b in range(B)]
    for _ in range(steps):
        out.append(np.stack([A[b] @ rng.standard_normal((m, n)) @ C[b].T for b in range(B)]))
    return out


def _check_step(pre, post, b, W_prev, W_new, G, lr, hp, t_prev, sch):
    st = O.OklsState(M=pre["M"][b], Sa=pre["Sa"][b], Sb=pre["Sb"][b], Pa=pre["Pa"][b],
                     Pb=pre["Pb"][b], t=t_prev)
    ost, Wo, Uo = O.shampoo_step(st, W_prev, G, lr, hp, root="exact")
    err = {"Sa": O.rel_fro(post["Sa"][b], ost.Sa), "Sb": O.rel_fro(post["Sb"][b], ost.Sb)}
    fresh = (t_prev % max(1, hp.root_every)) == 0
    for side in ("a", "b"):
        S_gpu, P_gpu = post["S" + side][b], post["P" + side][b]
        if fresh:
            err["P" + side] = O.rel_fro(P_gpu, O.quarter_root_exact(S_gpu, hp.ridge))
            err["P" + side + "_replay"] = O.rel_fro(P_gpu, O.quarter_root_chain(S_gpu, sch, hp.ridge, "replay"))
        else:
            err["P" + side] = err["P" + side + "_replay"] = O.rel_fro(P_gpu, pre["P" + side][b])
    decay = O.adamc_decay(lr, hp.peak, hp.weight_decay)
    U_gpu = ((1 - decay) * W_prev - W_new) / lr
    err["U"] = O.rel_fro(U_gpu, Uo)
    err["U_tf"] = O.rel_fro(U_gpu, post["Pa"][b] @ G @ post["Pb"][b])
    return err


@pytest.mark.parametrize("B,m,n,dtype", [(3, 200, 72, torch.float32), (2, 260, 260, torch.float32),
                                         (1, 130, 520, torch.float32), (2, 264, 136, torch.bfloat16)])
def test_teacher_forced_steps(B, m, n, dtype):
    steps = 4
    ob = _batch(B, m, n, param_dtype=dtype, eps=1e-6, weight_decay=0.01, lr=0.02)
    hp = hyper_of(ob)
    sch = O.cans_schedule(hp.ns_iters, hp.ns_lo)
    rng = np.random.default_rng(5)
    # |W| small next to the step, so bf16 rounding of W stays far below the bars
    W = torch.tensor(rng.standard_normal((B, m, n)) * 0.002, dtype=dtype, device="cuda")
    worst = {}
    for t, Gn in enumerate(_kron_grads(B, m, n, steps, seed=m + n), start=1):
        pre = snapshot(ob)
        Wp = W.double().cpu().numpy()
        G = torch.tensor(Gn, dtype=dtype, device="cuda")
        ob.step(W, G, hp.lr)
        assert ob.query_status() == 0
        post = snapshot(ob)
        Wn = W.double().cpu().numpy()
        Gd = G.double().cpu().numpy()
        for b in range(B):
            e = _check_step(pre, post, b, Wp[b], Wn[b], Gd[b], hp.lr, hp, t - 1, sch)
            for k, v in e.items():
                worst[k] = max(worst.get(k, 0.0), v)
        # the state's M is untouched in this mode
        assert not np.any(post["M"])
    print(f"shampoo {B}x{m}x{n} {dtype}", {k: f"{v:.2e}" for k, v in worst.items()})
    assert worst["Sa"] < 1e-3 and worst["Sb"] < 1e-3, worst
    assert worst["Pa"] < 1e-2 and worst["Pb"] < 1e-2, worst
    assert worst["Pa_replay"] < 3e-3 and worst["Pb_replay"] < 3e-3, worst
    u_tol = 3e-2 if dtype == torch.bfloat16 else 2e-2
    assert worst["U"] < u_tol, worst
    assert worst["U_tf"] < (2e-2 if dtype == torch.bfloat16 else 1e-2), worst
    ob.close()


def test_stale_quarter_roots():
    """root_every = 3: the roots of step 1 whiten steps 2 and 3 (bitwise the
    same state), step 4 refreshes them; the sums advance every step."""
    B, m, n = 2, 96, 160
    ob = _batch(B, m, n, eps=1e-6, weight_decay=0.0, lr=0.02, root_every=3)
    hp = hyper_of(ob)
    sch = O.cans_schedule(hp.ns_iters, hp.ns_lo)
    W = torch.zeros((B, m, n), device="cuda")
    prev = None
    for t, Gn in enumerate(_kron_grads(B, m, n, 4, seed=7), start=1):
        pre = snapshot(ob)
        Wp = W.double().cpu().numpy()
        G = torch.tensor(Gn, dtype=torch.float32, device="cuda")
        ob.step(W, G, hp.lr)
        assert ob.query_status() == 0
        post = snapshot(ob)
        if t in (2, 3):
            assert np.array_equal(post["Pa"], prev["Pa"]) and np.array_equal(post["Pb"], prev["Pb"])
            assert not np.allclose(post["Sa"], prev["Sa"])
        for b in range(B):
            e = _check_step(pre, post, b, Wp[b], W.double().cpu().numpy()[b], Gn[b], hp.lr, hp, t - 1, sch)
            assert e["Pa"] < 1e-2 and e["Pb"] < 1e-2 and e["U_tf"] < 1e-2, (t, e)
        prev = post
    ob.close()


def test_optimizer_class_matches_the_batch_api():
    from kronecker_factored_second_gb300.okls import OklsBatch, Shampoo
    torch.manual_seed(3)
    p = torch.nn.Parameter(torch.randn(2, 48, 80, device="cuda") * 0.02)
    W = p.detach().clone()
    opt = Shampoo([p], lr=0.05, eps=1e-6)
    ob = OklsBatch(2, 48, 80, lr=0.05, eps=1e-6, weight_decay=0.0, method="shampoo")
    for _ in range(3):
        g = torch.randn(2, 48, 80, device="cuda")
        p.grad = g.clone()
        opt.step()
        ob.step(W, g, 0.05)
    torch.cuda.synchronize()
    assert torch.equal(p.detach(), W)
    ob.close()


def test_failed_chain_keeps_previous_roots_with_their_scales():
    """OKLS mode without a ridge: the 64 x 64 left factor of a 64 x 16
    gradient has rank 16 at step 1, binary16 rounding gives it negative
    eigenvalues and the chain overflows (status bit 0x2); W and that factor's
    root stay as they were.  (The other factor's chain may finish and commit
    its new root; every root is committed together with its scale.)  With
    root_every = 2 the next step is a stale one: it must whiten with the
    roots in the state at their own scales, i.e. move W by exactly
    lr c_shape P_a N_2 P_b."""
    from kronecker_factored_second_gb300.okls import OklsBatch
    m, n = 64, 16
    ob = OklsBatch(1, m, n, ridge=0.0, root_every=2)
    hp = hyper_of(ob)
    rng = np.random.default_rng(11)
    W = torch.tensor(rng.standard_normal((1, m, n)) * 0.02, dtype=torch.float32, device="cuda")
    W0 = W.clone()
    G1 = torch.tensor(rng.standard_normal((1, m, n)), dtype=torch.float32, device="cuda")
    ob.step(W, G1, hp.lr)
    code, dev = ob.status_nothrow()
    assert dev & L.DEV_NONFINITE_ITER and code == L.OKLS_ERR_NONFINITE, (code, dev)
    assert torch.equal(W, W0)
    s1 = snapshot(ob)
    assert np.array_equal(s1["Pa"][0], np.eye(m))
    G2 = torch.tensor(rng.standard_normal((1, m, n)), dtype=torch.float32, device="cuda")
    Wp = W.double().cpu().numpy()[0]
    ob.step(W, G2, hp.lr)
    assert ob.query_status() == 0
    s2 = snapshot(ob)
    assert np.array_equal(s2["Pa"], s1["Pa"]) and np.array_equal(s2["Pb"], s1["Pb"])
    kappa = O.variance_correction(hp.beta1, 2)
    N2 = kappa * (hp.beta1 * s2["M"][0] + (1 - hp.beta1) * G2.double().cpu().numpy()[0])
    decay = O.adamc_decay(hp.lr, hp.peak, hp.weight_decay)
    want = -hp.lr * O.c_shape(m, n) * (s1["Pa"][0] @ N2 @ s1["Pb"][0])
    got = W.double().cpu().numpy()[0] - (1 - decay) * Wp
    assert O.rel_fro(got, want) < 3e-3, O.rel_fro(got, want)
    ob.close()
