"""Plain float64 restatement of the Online KL Shampoo step (test infrastructure).

Sources (page title, then section / equation):

* "Online KL Shampoo" (tilde-research release README), section "How it works":
  the KL-form factor EMAs, the fresh inverse roots, the two-sided whitening and
  the muP shape multiplier; bullet list under the title: 10-step "Scaled CANS
  Coupled Newton-Schulz", 27 FP16 GEMMs, FP32 accumulation, Nesterov momentum
  with variance correction, AdamC decoupled weight decay; section
  "Hyperparameters": defaults and the meaning of eps; section "Learning-rate
  schedule": lr_peak is the initial lr kept for the AdamC correction.
* "Shampoo" chapter of the optim-book (section "2 x 3 gradient by hand" and
  Problem 14): worked numbers used as pins.

Readings of points the pages leave open:

r1  P_0 = I at the first step (the EMAs use the previous roots).
r2  eps is added to both factors at initialisation (S_0 = eps*I) and at every
    update (+ eps*I).
r3  the factors are built from the raw gradient G, not from the momentum.
r4  Nesterov form: M_t = b1*M_{t-1} + (1-b1)*G_t,  N_t = b1*M_t + (1-b1)*G_t.
r5  "variance correction": N_t is divided by the standard deviation it would
    have for iid unit-variance gradients (``variance_correction``).
r6  AdamC: decoupled decay lr*wd*(lr/lr_peak)*W_{t-1}.
r7  W_t = W_{t-1} - decay - lr*c_shape*U_t, m = rows, n = cols.
r8  Chebyshev (CANS) coefficients are not printed: each step applies the odd
    cubic q(s) = a*s + b*s^3 that is the minimax approximation of 1 on the
    current interval [l, u] of sqrt-eigenvalues (``cans_schedule``).
r9  per-step scales are powers of two derived from the schedule alone.
r10 an optional relative ridge rho: the root is taken of S + rho*||S||_F*I.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Hyper", "OklsState", "c_shape", "variance_correction", "adamc_decay",
    "sym_power", "inv_root_exact", "inv_roots_exact", "cans_schedule", "ns_exponents",
    "ns_scalar_map", "ns_exact", "ns_matrix_float64", "f16", "split16",
    "ns_replay", "ns_replay_iteration", "factor_ema", "init_state",
    "okls_step", "okls_run", "rel_fro", "NS_HEADROOM", "NS_MARGIN",
    "quarter_root_exact", "quarter_root_chain", "shampoo_init", "shampoo_step",
    "SoapState", "soap_init", "soap_step", "eigenvectors_aligned",
    "nystrom_warm", "CleanState", "clean_init", "clean_step",
]

# Power-of-two headroom of the stored binary16 operands (reading r9): Y and T
# are stored times 2**12, Z times 2**(12 - z_k).  |Y| <= 2, |T| <= a_k <= 5.2
# and |Z| <= 2**z_k bound the entries, so the stored values stay below 2.2e4
# (binary16 max 65504) while typical entries, and the low halves of split
# pairs, stay above the subnormal range (6.1e-5).
NS_HEADROOM = 12
# Normalisation margin: Y_0 = S_reg / (||S||_F (1+rho) (1+2**-8)), so that the
# largest sqrt-eigenvalue sits strictly inside the first interval even after
# binary16 rounding of Y_0.
NS_MARGIN = 2.0 ** -8


@dataclass
class Hyper:
    """Hyperparameters; defaults from the 'Hyperparameters' table of the
    Online KL Shampoo README."""
    lr: float = 0.09434
    beta1: float = 0.9684
    beta2: float = 0.9482
    eps: float = 1e-9
    weight_decay: float = 0.0303
    lr_peak: float | None = None      # None -> lr (the initial lr is lr_peak)
    ns_iters: int = 10
    ns_lo: float = 1e-3               # l_0 of the coefficient schedule (r8)
    ridge: float = 0.0                # rho of reading r10
    variance_correction: bool = True  # reading r5
    eps_every_update: bool = True     # reading r2
    root_every: int = 1               # fresh roots at t = 1, 1+k, 1+2k, ... (1: every step)

    @property
    def peak(self) -> float:
        return self.lr if self.lr_peak is None else self.lr_peak


@dataclass
class OklsState:
    """Per-matrix state as listed under 'Hyperparameters' of the README: one
    (m,n) momentum and two copies each of the (m,m) and (n,n) shapes."""
    M: np.ndarray
    Sa: np.ndarray
    Sb: np.ndarray
    Pa: np.ndarray
    Pb: np.ndarray
    t: int = 0
    extra: dict = field(default_factory=dict)


# ---------------------------------------------------------------- scalars ---

def c_shape(m: int, n: int) -> float:
    """muP shape multiplier sqrt(m/n) / (sqrt(m) + sqrt(n)) ('How it works')."""
    return math.sqrt(m / n) / (math.sqrt(m) + math.sqrt(n))


def variance_correction(beta1: float, t: int) -> float:
    """kappa_t of reading r5.

    With M_0 = 0 and unrolled momentum,
        N_t = (1-b1) [ (1+b1) G_t + sum_{j=1}^{t-1} b1^(t-j+1) G_j ],
    so for iid unit-variance G_j its variance is
        v_t = (1-b1)^2 [ (1+b1)^2 + sum_{k=2}^{t} b1^(2k) ].
    The correction multiplies N_t by v_t^(-1/2).
    """
    if t < 1:
        raise ValueError("step index starts at 1")
    b = float(beta1)
    tail = 0.0
    for k in range(2, t + 1):
        tail += b ** (2 * k)
    v = (1.0 - b) ** 2 * ((1.0 + b) ** 2 + tail)
    return 1.0 / math.sqrt(v)


def adamc_decay(lr: float, lr_peak: float, wd: float) -> float:
    """Decoupled AdamC decay coefficient lr * wd * (lr / lr_peak) (r6)."""
    return lr * wd * (lr / lr_peak)


# ------------------------------------------------------------ exact roots ---

def _sym(S: np.ndarray) -> np.ndarray:
    S = np.asarray(S, dtype=np.float64)
    return 0.5 * (S + S.T)


def sym_power(S: np.ndarray, p: float, rcond: float | None = None) -> np.ndarray:
    """S^p of a symmetric PSD matrix by eigendecomposition.

    For p < 0, eigenvalues <= rcond * lambda_max are treated as zero (pseudo
    inverse), which is how a rank-deficient Shampoo factor is inverted in the
    optim-book's worked example.  rcond=None keeps every eigenvalue.
    """
    lam, Q = np.linalg.eigh(_sym(S))
    lam = np.maximum(lam, 0.0)
    out = np.zeros_like(lam)
    if p < 0:
        keep = lam > (0.0 if rcond is None else rcond * lam.max())
        out[keep] = lam[keep] ** p
    else:
        out = lam ** p
    return (Q * out) @ Q.T


def inv_root_exact(S: np.ndarray, ridge: float = 0.0) -> np.ndarray:
    """P = (S + ridge*||S||_F*I)^(-1/2), the exact root ('How it works':
    P_{a,t} = S_{a,t}^{-1/2}); ridge 0 is the plain root."""
    S = _sym(S)
    c = math.sqrt(float(np.sum(S * S)))
    return sym_power(S + ridge * c * np.eye(S.shape[0]), -0.5)


def inv_roots_exact(S: np.ndarray, ridges) -> list:
    """inv_root_exact(S, rho) for each rho in `ridges` from one
    eigendecomposition of S (for large factors, where eigh dominates)."""
    S = _sym(S)
    c = math.sqrt(float(np.sum(S * S)))
    lam, Q = np.linalg.eigh(S)
    out = []
    for rho in ridges:
        mu = np.maximum(lam + rho * c, 0.0)
        f = np.zeros_like(mu)
        keep = mu > 0.0
        f[keep] = mu[keep] ** -0.5
        out.append((Q * f) @ Q.T)
    return out


# -------------------------------------------------- Newton-Schulz schedule ---

def cans_schedule(iters: int = 10, lo: float = 1e-3, hi: float = 1.0):
    """Coefficients (a_k, b_k) and intervals [l_k, u_k] of reading r8.

    Coupled Newton-Schulz keeps Y_k, Z_k polynomials in S; with T_k = a I + b
    Z_k Y_k, an eigen-pair (y, z) of (Y_k, Z_k) moves to (y t, z t), t = a +
    b y z, so s = sqrt(y z) maps by the odd cubic q(s) = a s + b s^3 and the
    iteration converges when s -> 1 (then z -> lambda^(-1/2)).

    Each step picks the q minimising max |1 - q(s)| on [l, u].  Its error
    equioscillates at l, at the interior maximum s* = sqrt(-a/(3b)) and at u:
      q(l) = q(u)            gives  a = -b (u^2 + u l + l^2) = -b D,
      q(l) + q(s*) = 2       gives  a = 2 / (l u (u + l)/D + (2/3) sqrt(D/3)),
    and the next interval is [q(l), q(s*)].  For l = u = 1 this is the
    textbook (3/2, -1/2) step.
    """
    out = []
    l, u = float(lo), float(hi)
    for _ in range(iters):
        D = u * u + u * l + l * l
        a = 2.0 / (l * u * (u + l) / D + (2.0 / 3.0) * math.sqrt(D / 3.0))
        b = -a / D
        out.append((a, b, l, u))
        s_star = math.sqrt(D / 3.0)
        l, u = a * l + b * l ** 3, a * s_star + b * s_star ** 3
    return out


def ns_exponents(schedule) -> list[int]:
    """z_k = ceil(log2(prod_{j<k} a_j)), z_0 = 0 (reading r9).

    Every eigenvalue of Z_k is a product of factors t_j = a_j + b_j s^2 <= a_j
    (b_j < 0), so |Z_k| entries are bounded by 2**z_k; the stored operand is
    Z_k * 2**(headroom - z_k).  One entry per iterate k = 0..iters.
    """
    z = [0]
    prod = 1.0
    for (a, _b, _l, _u) in schedule:
        prod *= a
        z.append(int(math.ceil(math.log2(prod))))
    return z


def ns_scalar_map(mu: np.ndarray, schedule) -> tuple[np.ndarray, np.ndarray]:
    """Exact-arithmetic NS on eigenvalues mu of Y_0: returns (y_K, z_K)."""
    y = np.asarray(mu, dtype=np.float64).copy()
    z = np.ones_like(y)
    for (a, b, _l, _u) in schedule:
        t = a + b * y * z
        y, z = y * t, z * t
    return y, z


def _normaliser(S: np.ndarray, ridge: float) -> tuple[float, np.ndarray]:
    c = math.sqrt(float(np.sum(S * S)))
    cp = c * (1.0 + ridge) * (1.0 + NS_MARGIN)
    Y0 = (S + ridge * c * np.eye(S.shape[0])) / cp
    return cp, Y0


def ns_exact(S: np.ndarray, schedule, ridge: float = 0.0):
    """What the K-step iteration computes in exact arithmetic:
    P = Q diag(z_K(mu)) Q^T / sqrt(c'), root = Q diag(y_K(mu)) Q^T sqrt(c')."""
    S = _sym(S)
    cp, Y0 = _normaliser(S, ridge)
    mu, Q = np.linalg.eigh(Y0)
    y, z = ns_scalar_map(mu, schedule)
    return (Q * z) @ Q.T / math.sqrt(cp), (Q * y) @ Q.T * math.sqrt(cp)


def ns_matrix_float64(S: np.ndarray, schedule, ridge: float = 0.0):
    """The coupled matrix iteration in plain float64 (no rounding, no scales):
    T_k = a_k I + b_k Z_k Y_k; Y_{k+1} = Y_k T_k; Z_{k+1} = T_k Z_k."""
    S = _sym(S)
    d = S.shape[0]
    cp, Y = _normaliser(S, ridge)
    Z = np.eye(d)
    for (a, b, _l, _u) in schedule:
        T = a * np.eye(d) + b * (Z @ Y)
        Y, Z = Y @ T, T @ Z
    return Z / math.sqrt(cp), Y * math.sqrt(cp)


# ------------------------------------------------ binary16 replay of the NS ---

def f16(x) -> np.ndarray:
    """Round to IEEE binary16, round-to-nearest-even, back to float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def split16(x) -> tuple[np.ndarray, np.ndarray]:
    """hi = r16(x), lo = r16(x - hi): a pair of binary16 numbers whose sum
    carries about 22 significant bits (used by the split precision mode)."""
    hi = f16(x)
    return hi, f16(np.asarray(x, dtype=np.float64) - hi)


def _ns_consts(schedule, headroom=NS_HEADROOM):
    z = ns_exponents(schedule)
    return z, headroom, headroom, headroom


def _mm(A, B, acc32: bool):
    """A @ B in float64, or (acc32) with float32 operands and a float32
    result accumulated in the BLAS's own order (binary16 operands are exact
    in float32)."""
    if not acc32:
        return A @ B
    return (np.asarray(A, np.float32) @ np.asarray(B, np.float32)).astype(np.float64)


def _prod(A, B, split: bool, acc32: bool = False):
    """A @ B for stored operands; in split mode A, B are (hi, lo) pairs and
    the product keeps hi*hi + hi*lo + lo*hi (lo*lo is below the precision)."""
    if not split:
        return _mm(A, B, acc32)
    return _mm(A[0], B[0], acc32) + _mm(A[0], B[1], acc32) + _mm(A[1], B[0], acc32)


def ns_replay(S: np.ndarray, schedule, ridge: float = 0.0, rounding: bool = True,
              trace: bool = False, split_iters: int = 0, accumulate: str = "float64"):
    """Float64 replay of the coupled iteration as the GPU orders it, with every
    GEMM operand rounded to binary16 (rounding=False keeps float64 operands).

    Stored operands carry power-of-two scales (reading r9): Y^ = Y 2^h,
    Z^ = Z 2^(h - z_k), T^ = T 2^h.  Order of operations (27 products for 10
    steps, the count the README gives):
      k = 0:      Y0^ = r(Y_0 2^h);  T0^ = r(2^h a_0 I + b_0 Y0^)   (M_0 = Y_0)
                  Z1^ = r(T0^ 2^(-z_1));     Y1^ = r((Y0^ T0^) 2^-h)
      k = 1..K-1: T^  = r(2^h a_k I + b_k 2^(z_k - 2h + h) (Z^ Y^))
                  Y^' = r((Y^ T^) 2^-h)                  (not at k = K-1)
                  Z^' = r((T^ Z^) 2^(z_k - z_{k+1} - h))
      P = (T^_{K-1} Z^_{K-1}) 2^(z_{K-1} - 2h) / sqrt(c')
    This is the standard coupled order (M = Z Y, Y <- Y T, Z <- T Z).  Other
    orders that are equal in exact arithmetic (M = Y Z, Z <- Z T, mirroring a
    triangle) diverge under binary16 rounding, so the GPU keeps this one.

    split_iters > 0: the operands of iterations k < split_iters are (hi, lo)
    binary16 pairs (``split16``) and each product is hi*hi + hi*lo + lo*hi.

    accumulate="float32": every product is summed in float32 (in the BLAS's
    order) instead of float64.  Two float32 accumulation orders give two
    different chains: the distance between this replay and the float64 one
    measures how far accumulation order alone moves the result, the floor
    any fp32-accumulating implementation meets end to end.

    Returns dict with P, P_hat (binary16 copy of Z_K^), pi (P ~ pi * P_hat),
    c_prime, root (S^1/2 ~ Y_K sqrt(c') = (Y^_{K-1} T^_{K-1}) 2^(-2h) sqrt(c'))
    and, if trace, the lists Y, Z, T of stored iterates (index k is
    the operand of iteration k; Z[0] is None, Z_0 = I is never stored).
    """
    ident = (lambda x: np.asarray(x, dtype=np.float64))
    r = f16 if rounding else ident

    def rs(x, split):
        if split and rounding:
            return split16(x)
        if split:
            return (ident(x), np.zeros_like(x))
        return r(x)

    def val(x):
        return x[0] + x[1] if isinstance(x, tuple) else x

    S = _sym(S)
    d = S.shape[0]
    K = len(schedule)
    z, h, _, _ = _ns_consts(schedule)
    I = np.eye(d)
    cp, Y0 = _normaliser(S, ridge)
    Ys, Zs, Ts = [], [], []
    a32 = accumulate == "float32"
    if accumulate not in ("float64", "float32"):
        raise ValueError(accumulate)
    sp = split_iters > 0
    Yh = rs(Y0 * 2.0 ** h, sp)
    a0, b0 = schedule[0][0], schedule[0][1]
    Th = rs(2.0 ** h * a0 * I + b0 * val(Yh), sp)
    sp1 = split_iters > 1
    Zh = rs(val(Th) * 2.0 ** (-z[1]), sp1)
    Ys.append(Yh); Zs.append(None); Ts.append(Th)
    Yh = rs(_prod(Yh, Th, sp, a32) * 2.0 ** -h, sp1)
    Zacc = None
    for k in range(1, K):
        spk = split_iters > k
        spn = split_iters > k + 1
        a, b = schedule[k][0], schedule[k][1]
        Ys.append(Yh); Zs.append(Zh)
        Mfac = b * 2.0 ** (z[k] - h)
        Th = rs(2.0 ** h * a * I + Mfac * _prod(Zh, Yh, spk, a32), spk)
        Ts.append(Th)
        Zacc = _prod(Th, Zh, spk, a32)
        Yacc = _prod(Yh, Th, spk, a32)
        if k < K - 1:
            Yh = rs(Yacc * 2.0 ** -h, spn)
            Zh = rs(Zacc * 2.0 ** (z[k] - z[k + 1] - h), spn)
    k = K - 1
    P = Zacc * 2.0 ** (z[k] - 2 * h) / math.sqrt(cp)
    P_hat = r(Zacc * 2.0 ** (z[k] - z[k + 1] - h))
    pi = 2.0 ** (z[K] - h) / math.sqrt(cp)
    # the square root S^1/2 ~ Y_K sqrt(c'), formed from the last (Y^, T^)
    root = Yacc * 2.0 ** (-2 * h) * math.sqrt(cp)
    out = {"P": P, "P_hat": P_hat, "pi": pi, "c_prime": cp, "root": root}
    if trace:
        out.update(Y=Ys, Z=Zs, T=Ts)
    return out


def ns_replay_iteration(k: int, Yh: np.ndarray, Zh: np.ndarray, schedule,
                        rounding: bool = True):
    """One step k >= 1 of ``ns_replay`` (binary16 operands) from given stored
    iterates (Y^_k, Z^_k): returns (T^_k, Y^_{k+1} or None, Z^_{k+1}).  Used
    for the per-iteration teacher-forced comparison with the GPU iterates."""
    r = f16 if rounding else (lambda x: np.asarray(x, dtype=np.float64))
    K = len(schedule)
    z, h, _, _ = _ns_consts(schedule)
    d = Yh.shape[0]
    a, b = schedule[k][0], schedule[k][1]
    Th = r(2.0 ** h * a * np.eye(d) + b * 2.0 ** (z[k] - h) * (Zh @ Yh))
    Zn = r((Th @ Zh) * 2.0 ** (z[k] - z[k + 1] - h))
    Yn = r((Yh @ Th) * 2.0 ** -h) if k < K - 1 else None
    return Th, Yn, Zn


# ----------------------------------------------------------- the OKLS step ---

def factor_ema(S_prev: np.ndarray, X: np.ndarray, beta2: float, count: int,
               eps: float) -> np.ndarray:
    """S <- beta2 S + (1-beta2)/count * X X^T + eps I  ('How it works').

    Left factor: X = G P_b, count = n.  Right factor: X = (P_a G)^T, count = m.
    """
    X = np.asarray(X, dtype=np.float64)
    d = X.shape[0]
    return beta2 * S_prev + (1.0 - beta2) / count * (X @ X.T) + eps * np.eye(d)


def init_state(m: int, n: int, hp: Hyper) -> OklsState:
    """M_0 = 0, S_0 = eps I (README: eps is added at factor initialisation),
    P_0 = I (reading r1)."""
    return OklsState(
        M=np.zeros((m, n)),
        Sa=hp.eps * np.eye(m), Sb=hp.eps * np.eye(n),
        Pa=np.eye(m), Pb=np.eye(n), t=0)


def okls_step(state: OklsState, W: np.ndarray, G: np.ndarray, lr: float,
              hp: Hyper, root: str = "exact"):
    """One OKLS step for one matrix in float64.  Returns (new_state, W_new, U).

    root: "exact" (eigendecomposition), "ns_exact" (the K-step polynomial in
    exact arithmetic) or "replay" (binary16 replay of the GPU iteration).
    """
    G = np.asarray(G, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    m, n = G.shape
    t = state.t + 1
    b1, b2 = hp.beta1, hp.beta2
    # momentum, reading r4/r5
    M = b1 * state.M + (1.0 - b1) * G
    kappa = variance_correction(b1, t) if hp.variance_correction else 1.0
    N = kappa * (b1 * M + (1.0 - b1) * G)
    # factor EMAs with the previous roots (r3; 'How it works')
    eps_upd = hp.eps if hp.eps_every_update else 0.0
    Sa = factor_ema(state.Sa, G @ state.Pb, b2, n, eps_upd)
    Sb = factor_ema(state.Sb, (state.Pa @ G).T, b2, m, eps_upd)
    # fresh roots in the same step ('How it works'); with root_every = k > 1
    # only at t = 1, 1+k, ... and the previous roots in between
    if (t - 1) % max(1, hp.root_every) != 0:
        Pa, Pb = state.Pa, state.Pb
    elif root == "exact":
        Pa, Pb = inv_root_exact(Sa, hp.ridge), inv_root_exact(Sb, hp.ridge)
    elif root == "ns_exact":
        sch = cans_schedule(hp.ns_iters, hp.ns_lo)
        Pa, Pb = ns_exact(Sa, sch, hp.ridge)[0], ns_exact(Sb, sch, hp.ridge)[0]
    elif root == "replay":
        sch = cans_schedule(hp.ns_iters, hp.ns_lo)
        Pa = ns_replay(Sa, sch, hp.ridge)["P"]
        Pb = ns_replay(Sb, sch, hp.ridge)["P"]
    else:
        raise ValueError(root)
    # two-sided whitening and update, readings r6/r7
    U = Pa @ N @ Pb
    decay = adamc_decay(lr, hp.peak, hp.weight_decay)
    W_new = W - decay * W - lr * c_shape(m, n) * U
    return OklsState(M=M, Sa=Sa, Sb=Sb, Pa=Pa, Pb=Pb, t=t), W_new, U


def okls_run(W0: np.ndarray, grads, hp: Hyper, lrs=None, root: str = "exact"):
    """Free-running OKLS over a gradient sequence; returns (state, W, Us)."""
    m, n = np.asarray(W0).shape
    st = init_state(m, n, hp)
    W = np.asarray(W0, dtype=np.float64)
    Us = []
    for i, G in enumerate(grads):
        lr = hp.lr if lrs is None else lrs[i]
        st, W, U = okls_step(st, W, G, lr, hp, root=root)
        Us.append(U)
    return st, W, Us


# ---------------------------------------------------- classic Shampoo ---
#
# "Shampoo" chapter of the optim-book, sections "2 x 3 gradient by hand" and
# Problem 14: the row factor L and the column factor R are plain sums of
# G G^T and G^T G over the steps, and the step multiplies the gradient by
# L^-1/4 on the left and R^-1/4 on the right (the -1/4 makes the step
# invariant to the scale of G).  Readings of what the chapter leaves open:
#   s1  L_0 = R_0 = eps I (the README's eps at factor initialisation); no eps
#       at later steps.
#   s2  the step is W <- W - decay - lr U with U = L^-1/4 G R^-1/4: no
#       momentum, no shape multiplier; decay is the same decoupled term as
#       the OKLS step (weight_decay = 0 gives the chapter's plain step).
#   s3  L^-1/4 = (L^1/2)^-1/2: the square root from one Newton-Schulz chain
#       (ridge rho on L) is the input of a second chain without a ridge; its
#       condition number is at most sqrt((1+rho)/rho).  The exact reference is
#       (L + rho ||L||_F I)^-1/4.
#   s4  roots are refreshed every root_every steps like the OKLS roots.

def quarter_root_exact(S: np.ndarray, ridge: float = 0.0) -> np.ndarray:
    """(S + rho ||S||_F I)^-1/4 by eigendecomposition (reading s3)."""
    S = _sym(S)
    c = math.sqrt(float(np.sum(S * S)))
    return sym_power(S + ridge * c * np.eye(S.shape[0]), -0.25)


def quarter_root_chain(S: np.ndarray, schedule, ridge: float = 0.0,
                       mode: str = "ns_exact", split_iters: int = 0) -> np.ndarray:
    """S^-1/4 as two chained K-step Newton-Schulz runs (reading s3).

    mode "ns_exact": both chains in exact arithmetic (``ns_exact``).
    mode "replay":   both chains as the binary16 replay (``ns_replay``); the
                     square root between them is held in float32, as the GPU
                     keeps it.
    """
    if mode == "ns_exact":
        root = ns_exact(S, schedule, ridge)[1]
        return ns_exact(root, schedule, 0.0)[0]
    if mode == "replay":
        root = ns_replay(S, schedule, ridge, split_iters=split_iters)["root"]
        root = root.astype(np.float32).astype(np.float64)
        return ns_replay(root, schedule, 0.0, split_iters=split_iters)["P"]
    raise ValueError(mode)


def shampoo_init(m: int, n: int, hp: Hyper) -> OklsState:
    """L_0 = eps I, R_0 = eps I (reading s1), roots I; M is unused."""
    return OklsState(
        M=np.zeros((m, n)),
        Sa=hp.eps * np.eye(m), Sb=hp.eps * np.eye(n),
        Pa=np.eye(m), Pb=np.eye(n), t=0)


def shampoo_step(state: OklsState, W: np.ndarray, G: np.ndarray, lr: float,
                 hp: Hyper, root: str = "exact"):
    """One classic Shampoo step for one matrix in float64 (Sa = L, Sb = R,
    Pa = L^-1/4, Pb = R^-1/4).  Returns (new_state, W_new, U).

    root: "exact" (eigendecomposition), "ns_exact" (two chained K-step
    polynomials in exact arithmetic) or "replay" (two chained binary16
    replays of the GPU iteration).
    """
    G = np.asarray(G, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    m, n = G.shape
    t = state.t + 1
    L = state.Sa + G @ G.T
    R = state.Sb + G.T @ G
    if (t - 1) % max(1, hp.root_every) != 0:
        Pa, Pb = state.Pa, state.Pb
    elif root == "exact":
        Pa, Pb = quarter_root_exact(L, hp.ridge), quarter_root_exact(R, hp.ridge)
    elif root in ("ns_exact", "replay"):
        sch = cans_schedule(hp.ns_iters, hp.ns_lo)
        Pa = quarter_root_chain(L, sch, hp.ridge, root)
        Pb = quarter_root_chain(R, sch, hp.ridge, root)
    else:
        raise ValueError(root)
    U = Pa @ G @ Pb
    decay = adamc_decay(lr, hp.peak, hp.weight_decay)
    W_new = W - decay * W - lr * U
    return OklsState(M=state.M, Sa=L, Sb=R, Pa=Pa, Pb=Pb, t=t), W_new, U


# ------------------------------------------------------- SOAP (eigenbasis Adam) ---
#
# Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
# Sketching", Appendix C, Algorithm 4 (SOAP), with the KPOP page's section on
# running Adam in the Kronecker-factored eigenbasis for the Adam details.
# Per step: rotate G and the momentum M (kept in the original space) into the
# eigenbases Q_L, Q_R of the factors L, R; run Adam there with the second
# moment V kept in the rotated space; rotate the normalised step back; then
# update L, R, and every f steps refresh Q_L, Q_R.  Readings:
#   p1  "run Adam on G'": standard Adam, both moments bias-corrected,
#       N' = (M' / (1 - b1^t)) / (sqrt(V / (1 - b2^t)) + eps) (the KPOP page's
#       formula; the Clean listing prints the correction on V).
#   p2  Q_L = I, Q_R = I before the first refresh (L = R = 0).
#   p3  Eigenvectors(L, Q_L): the eigenvectors of L with eigenvalues in
#       decreasing order, each column's sign chosen so it has a non-negative
#       inner product with the same column of the previous basis (the sign
#       alignment of the Clean page's Algorithm 3).
#   p4  the refresh happens at the end of steps t with t % f == 0; V is kept
#       as it is across a refresh.
#   p5  W <- W - decay - lr N, decay the same decoupled term as OKLS (zero
#       with weight_decay = 0, the listing's plain step).

@dataclass
class SoapState:
    M: np.ndarray    # m x n, original space
    V: np.ndarray    # m x n, eigenbasis
    L: np.ndarray    # m x m
    R: np.ndarray    # n x n
    QL: np.ndarray   # m x m
    QR: np.ndarray   # n x n
    t: int = 0


def soap_init(m: int, n: int) -> SoapState:
    return SoapState(M=np.zeros((m, n)), V=np.zeros((m, n)), L=np.zeros((m, m)), R=np.zeros((n, n)),
                     QL=np.eye(m), QR=np.eye(n), t=0)


def eigenvectors_aligned(S: np.ndarray, Q_prev: np.ndarray) -> np.ndarray:
    """Reading p3: eigenvectors of the symmetric S, eigenvalues decreasing,
    column signs aligned with the previous basis."""
    w, Q = np.linalg.eigh(_sym(S))
    Q = Q[:, ::-1]
    s = np.sign(np.sum(Q * Q_prev, axis=0))
    s[s == 0] = 1.0
    return Q * s


def soap_step(state: SoapState, W: np.ndarray, G: np.ndarray, lr: float, beta1: float, beta2: float,
              eps: float, f: int, weight_decay: float = 0.0, lr_peak: float | None = None):
    """One SOAP step for one matrix in float64.  Returns (new_state, W_new, N)."""
    G = np.asarray(G, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    t = state.t + 1
    QL, QR = state.QL, state.QR
    Gr = QL.T @ G @ QR
    M = beta1 * state.M + (1.0 - beta1) * G
    Mr = QL.T @ M @ QR
    V = beta2 * state.V + (1.0 - beta2) * Gr * Gr
    Nr = (Mr / (1.0 - beta1 ** t)) / (np.sqrt(V / (1.0 - beta2 ** t)) + eps)
    N = QL @ Nr @ QR.T
    decay = adamc_decay(lr, lr if lr_peak is None else lr_peak, weight_decay)
    W_new = W - decay * W - lr * N
    L = beta2 * state.L + (1.0 - beta2) * (G @ G.T)
    R = beta2 * state.R + (1.0 - beta2) * (G.T @ G)
    if t % max(1, f) == 0:
        QL = eigenvectors_aligned(L, QL)
        QR = eigenvectors_aligned(R, QR)
    return SoapState(M=M, V=V, L=L, R=R, QL=QL, QR=QR, t=t), W_new, N


# ------------------------------------------------------------- Clean (Nystrom) ---
#
# Page "Clean: Second-order LLM Training at Linear Memory Cost via Nystrom
# Sketching": Algorithm 1 (the step), Eqn. (8) (the sketch of the factor
# without forming it), Eqns. (10)-(13) and Table 1 (the four blocks and their
# moments), Eqns. (14)-(15) (moving the moments to refreshed bases), Eqn. (16)
# (the update), Appendix A Algorithm 3 (warm-started Nystrom with subspace
# iteration).  Readings:
#   c1  Algorithm 3 orthonormalises the starting sketch in both branches
#       (warm start [U_prev, Psi] and cold start) with a thin QR before the
#       power iterations.
#   c2  eps(x) is the spacing of binary64 numbers at x: 2^(floor(log2 x) - 52);
#       norm(Y, 2) is the spectral norm.
#   c3  Y_nu / C is right division, Y_nu C^-1, with C the upper Cholesky
#       factor (C^T C = (B + B^T)/2).
#   c4  the Gaussian draws Psi are inputs (m x p with a warm start, m x (r+p)
#       at the first refresh); thin QR takes R with a non-negative diagonal.
#   c5  the factor sketched at a refresh is b2 U Lambda U^T + (1-b2) G G^T
#       with the previous refresh's factors, (1-b2) G G^T at the first one.
#   c6  the moments use the step count t of the whole run for their bias
#       corrections; the pooled second moments are sums (1^T (G_A)^2,
#       (G_B)^2 1, ||C||_F^2) as printed, bias-corrected like V.
#   c7  W <- W - alpha lr G~ (no weight decay in the listing); alpha = 1.

def _qr_pos(X: np.ndarray) -> np.ndarray:
    """Thin QR with a non-negative diagonal of R (reading c4)."""
    Q, R = np.linalg.qr(X)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s


def _eps64(x: float) -> float:
    """Spacing of binary64 numbers at x (reading c2)."""
    return 0.0 if x == 0.0 else 2.0 ** (math.floor(math.log2(abs(x))) - 52)


def nystrom_warm(apply_A, r: int, p: int, q: int, U_prev, Psi: np.ndarray):
    """Algorithm 3: rank-r Nystrom approximation [U, Lambda] of the PSD
    operator apply_A (X -> A X), warm-started at U_prev (or None)."""
    Omega = np.hstack([U_prev, Psi]) if U_prev is not None else Psi
    Omega = _qr_pos(Omega)
    for _ in range(q):
        Omega = _qr_pos(apply_A(Omega))
    Y = apply_A(Omega)
    nu = _eps64(float(np.linalg.norm(Y, 2)))
    Yn = Y + nu * Omega
    B = Omega.T @ Yn
    C = np.linalg.cholesky(0.5 * (B + B.T)).T          # upper: C^T C = (B + B^T)/2
    U, sig, _vt = np.linalg.svd(np.linalg.solve(C.T, Yn.T).T, full_matrices=False)
    lam = np.maximum(0.0, sig ** 2 - nu)
    U, lam = U[:, :r], lam[:r]
    if U_prev is not None:
        s = np.sign(np.sum(U * U_prev, axis=0))
        s[s == 0] = 1.0
        U = U * s
    return U, lam


@dataclass
class CleanState:
    UL: np.ndarray | None = None   # m x r
    lamL: np.ndarray | None = None
    UR: np.ndarray | None = None   # n x r
    lamR: np.ndarray | None = None
    M: np.ndarray | None = None    # r x r (Main)
    V: np.ndarray | None = None
    MA: np.ndarray | None = None   # m x r (block A)
    vA: np.ndarray | None = None   # r
    MB: np.ndarray | None = None   # r x n (block B)
    vB: np.ndarray | None = None   # r
    vC: float = 0.0                # block C
    t: int = 0


def clean_init(m: int, n: int, r: int) -> CleanState:
    return CleanState(M=np.zeros((r, r)), V=np.zeros((r, r)), MA=np.zeros((m, r)), vA=np.zeros(r),
                      MB=np.zeros((r, n)), vB=np.zeros(r), vC=0.0, t=0)


def clean_step(state: CleanState, W: np.ndarray, G: np.ndarray, lr: float, beta1: float, beta2: float,
               eps: float, r: int, p: int, q: int, T: int, psiL=None, psiR=None, alpha: float = 1.0,
               bases=None):
    """One Clean step for one matrix in float64 (Algorithm 1).  psiL, psiR
    are the Gaussian draws of a refresh step.  `bases` = (U_L, Lambda_L,
    U_R, Lambda_R), when given, stands in for Algorithm 3's output at a
    refresh (teacher forcing: the rest of the step then runs on those
    bases).  Returns (state, W_new, G~)."""
    G = np.asarray(G, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    m, n = G.shape
    t = state.t + 1
    st = CleanState(**{k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in state.__dict__.items()})
    st.t = t
    if (t - 1) % T == 0:
        def aL(X, U=st.UL, lam=st.lamL):
            out = (1.0 - beta2) * (G @ (G.T @ X))
            return out + beta2 * (U @ (lam[:, None] * (U.T @ X))) if U is not None else out

        def aR(X, U=st.UR, lam=st.lamR):
            out = (1.0 - beta2) * (G.T @ (G @ X))
            return out + beta2 * (U @ (lam[:, None] * (U.T @ X))) if U is not None else out
        if bases is None:
            ULn, lamLn = nystrom_warm(aL, r, p, q, st.UL, psiL)
            URn, lamRn = nystrom_warm(aR, r, p, q, st.UR, psiR)
        else:
            ULn, lamLn, URn, lamRn = (np.asarray(x, dtype=np.float64) for x in bases)
        if st.UL is not None:
            # Eqns. (14)-(15): moments into the new bases
            OL = ULn.T @ st.UL            # r x r: new^T old
            OR = st.UR.T @ URn            # r x r: old^T new
            PLn = np.eye(m) - ULn @ ULn.T
            PRn = np.eye(n) - URn @ URn.T
            st.M = OL @ st.M @ OR
            st.MA = PLn @ st.MA @ OR
            st.MB = OL @ st.MB @ PRn
            st.vA = st.vA @ (OR * OR)
            st.vB = (OL * OL) @ st.vB
        st.UL, st.lamL, st.UR, st.lamR = ULn, lamLn, URn, lamRn
    UL, UR = st.UL, st.UR
    PL = np.eye(m) - UL @ UL.T
    PR = np.eye(n) - UR @ UR.T
    S = UL.T @ G @ UR
    GA = PL @ G @ UR
    GB = UL.T @ G @ PR
    C = PL @ G @ PR
    st.M = beta1 * st.M + (1.0 - beta1) * S
    st.V = beta2 * st.V + (1.0 - beta2) * S * S
    st.MA = beta1 * st.MA + (1.0 - beta1) * GA
    st.vA = beta2 * st.vA + (1.0 - beta2) * np.sum(GA * GA, axis=0)
    st.MB = beta1 * st.MB + (1.0 - beta1) * GB
    st.vB = beta2 * st.vB + (1.0 - beta2) * np.sum(GB * GB, axis=1)
    st.vC = beta2 * st.vC + (1.0 - beta2) * float(np.sum(C * C))
    c1, c2 = 1.0 - beta1 ** t, 1.0 - beta2 ** t
    main = (st.M / c1) / (np.sqrt(st.V / c2) + eps)
    blkA = (st.MA / c1) / (np.sqrt(st.vA / c2)[None, :] + eps)
    blkB = (st.MB / c1) / (np.sqrt(st.vB / c2)[:, None] + eps)
    blkC = C / (math.sqrt(st.vC / c2) + eps)
    Gt = UL @ main @ UR.T + blkA @ UR.T + UL @ blkB + blkC
    return st, W - alpha * lr * Gt, Gt


def rel_fro(A: np.ndarray, B: np.ndarray) -> float:
    """||A - B||_F / ||B||_F."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    nb = float(np.linalg.norm(B))
    return float(np.linalg.norm(A - B)) / (nb if nb > 0 else 1.0)
