"""Shared helpers of the GPU parity tests (teacher-forced oracle comparison)."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
from kronecker_factored_second_gb300 import _lib as L

PARTS = [("M", L.STATE_M), ("Sa", L.STATE_SA), ("Sb", L.STATE_SB), ("Pa", L.STATE_PA),
         ("Pb", L.STATE_PB)]


def snapshot(ob) -> dict:
    """All state parts of an OklsBatch as float64 numpy arrays."""
    torch.cuda.synchronize()
    return {k: ob.get_state(p).double().cpu().numpy() for k, p in PARTS}


def kappa_f(S: np.ndarray, ridge: float = 0.0) -> float:
    """||S||_F / lambda_min of the ridged factor S + ridge ||S||_F I: the
    spread the Newton-Schulz chain must cover."""
    S = 0.5 * (S + S.T)
    c = float(np.linalg.norm(S))
    lam = np.linalg.eigvalsh(S) + ridge * c
    return float(c / max(lam.min(), 1e-300 * max(c, 1e-300)))


def hyper_of(ob, lr=None) -> O.Hyper:
    c = ob.cfg
    return O.Hyper(lr=float(c.lr_peak) if lr is None else lr, beta1=float(c.beta1),
                   beta2=float(c.beta2), eps=float(c.eps), weight_decay=float(c.weight_decay),
                   lr_peak=float(c.lr_peak), ns_iters=int(c.ns_iters), ns_lo=float(c.ns_lo),
                   ridge=float(c.ridge), variance_correction=bool(c.variance_correction),
                   eps_every_update=bool(c.eps_every_update), root_every=max(1, int(c.root_every)))


def compare_step(pre: dict, post: dict, b: int, W_prev: np.ndarray, W_new: np.ndarray,
                 G: np.ndarray, lr: float, hp: O.Hyper, t_prev: int) -> dict:
    """Teacher-forced comparison of matrix b of one step.  Returns the errors."""
    st = O.OklsState(M=pre["M"][b], Sa=pre["Sa"][b], Sb=pre["Sb"][b], Pa=pre["Pa"][b],
                     Pb=pre["Pb"][b], t=t_prev)
    ost, Wo, Uo = O.okls_step(st, W_prev, G, lr, hp, root="exact")
    m, n = G.shape
    out = {}
    out["M"] = O.rel_fro(post["M"][b], ost.M)
    out["Sa"] = O.rel_fro(post["Sa"][b], ost.Sa)
    out["Sb"] = O.rel_fro(post["Sb"][b], ost.Sb)
    sch = O.cans_schedule(hp.ns_iters, hp.ns_lo)
    fresh = (t_prev % max(1, hp.root_every)) == 0
    for side in ("a", "b"):
        S_gpu = post["S" + side][b]
        P_gpu = post["P" + side][b]
        if fresh:
            ref = O.ns_exact(S_gpu, sch, hp.ridge)[0]
            out["P" + side] = O.rel_fro(P_gpu, ref)
            out["P" + side + "_exact"] = O.rel_fro(P_gpu, O.inv_root_exact(S_gpu, hp.ridge))
        else:
            # a step that keeps the roots: P must be the previous P
            out["P" + side] = out["P" + side + "_exact"] = O.rel_fro(P_gpu, pre["P" + side][b])
        out["kf_" + side] = kappa_f(S_gpu, hp.ridge)
    decay = O.adamc_decay(lr, hp.peak, hp.weight_decay)
    c = O.c_shape(m, n)
    dW_gpu = W_new - (1 - decay) * W_prev
    U_gpu = -dW_gpu / (lr * c) if lr > 0 else None
    # whitening with the GPU's own roots (checks N and the two GEMMs)
    kappa = O.variance_correction(hp.beta1, t_prev + 1) if hp.variance_correction else 1.0
    N = kappa * (hp.beta1 * ost.M + (1 - hp.beta1) * G)
    U_tf = post["Pa"][b] @ N @ post["Pb"][b]
    if U_gpu is not None:
        out["U"] = O.rel_fro(U_gpu, Uo)
        out["U_tf"] = O.rel_fro(U_gpu, U_tf)
    out["dW"] = O.rel_fro(dW_gpu, Wo - (1 - decay) * W_prev)
    return out


def spd(d: int, cond: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    w = np.exp(rng.uniform(0.0, math.log(cond), d))
    w[0], w[-1] = 1.0, cond
    return (Q * w) @ Q.T
