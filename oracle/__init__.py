"""Float64 CPU oracle for the Online KL Shampoo (OKLS) preconditioner step,
the classic Shampoo step it refines, SOAP (Adam in the factors' eigenbasis)
and Clean (Nyström low-rank factors with block-wise Adam).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code, table or constant generator with
the CUDA library; where both sides need the same number (the Newton-Schulz
coefficient schedule, the momentum variance correction) each side derives it
independently from the same written definition.

Parity status per function (the pins live in ``tests/test_oracle_pins.py``):

* ``sym_power`` / ``inv_root_exact``      pinned (Shampoo 2x3 hand example,
  Problem 14, eigen-identities).
* ``cans_schedule``                        pinned (textbook Newton-Schulz special
  case, brute-force minimax, equioscillation).
* ``ns_exact``, ``ns_replay``             pinned (scalar-polynomial identity,
  convergence bound, fp16 rounding checks).
* ``factor_ema``                           pinned (hand example L = G G^T,
  brute-force loops).
* ``okls_step`` / ``okls_run``             pinned (square fixed-gradient polar
  limit, descent sign, closed-form weight decay, the Nesterov combination
  kappa_t (1 - b1^(t+1)) G of a constant gradient recovered through the
  step's roots).
* ``shampoo_step``                         pinned (the page's 2x3 gradient fed 1,
  4 and 100 times: step singular values 1 / 0.5 / 0.1; scale invariance of
  Problem 14; brute-force factor sums).
* ``quarter_root_exact``, ``quarter_root_chain``  pinned (chained exact chains
  equal the eigendecomposition quarter root, P^4 S = I; the replay's square
  root equals the float64 iteration's).
* ``soap_step``, ``eigenvectors_aligned``   pinned (no refresh: textbook Adam by
  entry loops; fixed bases: rotated Adam; eigenvector order and signs;
  refresh schedule).  The readings of the bias correction, the initial bases
  and the eigenvector signs follow the pages' listings; no printed values.
* ``nystrom_warm``, ``clean_step``          pinned (exactly low-rank operators
  recovered, with and without warm start; power iterations track the top
  eigenpairs; the four blocks partition G; pooled moments by entry loops;
  full-rank bases reduce to rotated Adam; unchanged bases leave the moments
  in place).  Readings c1-c7 in the module; no printed values.
* ``variance_correction``                  pinned by Monte Carlo against its
  definition (variance of the Nesterov combination for iid unit gradients);
  the *choice* of this reading is not printed on the pages.
* AdamC correction factor lr/lr_peak       parity unpinned by the pages (a
  closed-form scalar whose reading the pages name without a formula; the
  G = 0 decay test fixes its arithmetic, not the reading).
"""

from .okls_oracle import *  # noqa: F401,F403
