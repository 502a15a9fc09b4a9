"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the header declares, validates its arguments, and computes the
same coefficient schedule as the oracle from the same definition."""

import ctypes
import os

import numpy as np
import pytest

from kronecker_factored_second_gb300 import _lib as L


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from kronecker_factored_second_gb300.build import build_library
        build_library()
    return L.lib()


def test_library_exports_every_header_function(lib):
    names = L.header_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name
    assert lib.okls_abi_version() == 3


def test_header_names_match_binding():
    assert set(L.header_functions()) == set(L._SIGS)


def test_config_defaults_are_readme_values(lib):
    c = L.config_default(3, 128, 64)
    assert (c.batch, c.m, c.n) == (3, 128, 64)
    assert abs(c.lr_peak - 0.09434) < 1e-7 and abs(c.beta1 - 0.9684) < 1e-7
    assert abs(c.beta2 - 0.9482) < 1e-7 and abs(c.eps - 1e-9) < 1e-15
    assert abs(c.weight_decay - 0.0303) < 1e-7 and c.ns_iters == 10
    assert c.variance_correction == 1 and c.eps_every_update == 1


def test_state_bytes_layout(lib):
    c = L.config_default(2, 128, 64)
    sb, wb = L.state_bytes(c)
    # M + S_a + S_b + P_a + P_b in fp32 (each block 256-byte aligned)
    want = 4 * 2 * (128 * 64 + 2 * 128 * 128 + 2 * 64 * 64)
    assert want <= sb <= want + 5 * 256
    assert wb > 0
    c.ns_split_iters = 3
    _, wb3 = L.state_bytes(c)
    assert wb3 > wb


@pytest.mark.parametrize("field,value", [
    ("batch", 0), ("m", 0), ("n", -1), ("beta1", 1.0), ("beta2", -0.1), ("eps", -1.0),
    ("weight_decay", float("nan")), ("ns_iters", 1), ("ns_split_iters", 11), ("ns_lo", 0.0),
    ("ridge", -1.0), ("lr_peak", 0.0), ("param_dtype", 7), ("m", 1 << 20)])
def test_invalid_configs_rejected(lib, field, value):
    c = L.config_default(1, 64, 32)
    setattr(c, field, value)
    s, w = ctypes.c_size_t(), ctypes.c_size_t()
    code = lib.okls_state_bytes(ctypes.byref(c), ctypes.byref(s), ctypes.byref(w))
    assert code in (L.OKLS_ERR_INVALID_ARG, L.OKLS_ERR_UNSUPPORTED)
    assert L.last_error()


def test_reserved_fields_must_be_zero(lib):
    c = L.config_default(1, 64, 32)
    c.reserved[2] = 1
    assert lib.okls_state_bytes(ctypes.byref(c), None, None) == L.OKLS_ERR_INVALID_ARG


def test_null_arguments(lib):
    assert lib.okls_state_bytes(None, None, None) == L.OKLS_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    c = L.config_default(1, 64, 32)
    assert lib.okls_create(ctypes.byref(c), None, 0, None, 0, ctypes.byref(h)) == L.OKLS_ERR_INVALID_ARG
    assert lib.okls_step(None, None, None, ctypes.c_float(0.1), None) == L.OKLS_ERR_INVALID_ARG
    assert lib.okls_destroy(None) == L.OKLS_OK
    assert lib.okls_ns_schedule(0, 1e-3, None, None, None) == L.OKLS_ERR_INVALID_ARG
    assert lib.okls_set_wait_limit(None, 0, -1) == L.OKLS_ERR_INVALID_ARG


def test_schedule_matches_oracle_definition(lib):
    """The library and the oracle derive the coefficients independently from
    the same minimax definition; they must agree to rounding."""
    import oracle as O
    a, b, z = L.ns_schedule(10, 1e-3)
    sch = O.cans_schedule(10, 1e-3)
    assert np.allclose(a, [s[0] for s in sch], rtol=1e-13)
    assert np.allclose(b, [s[1] for s in sch], rtol=1e-13)
    assert z == O.ns_exponents(sch)
    a1, b1, _ = L.ns_schedule(1, 1.0)
    assert abs(a1[0] - 1.5) < 1e-15 and abs(b1[0] + 0.5) < 1e-15


def test_create_without_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = L.config_default(1, 64, 32)
    sb, wb = L.state_bytes(c)
    buf = ctypes.create_string_buffer(sb + wb + 512)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    h = ctypes.c_void_p()
    code = lib.okls_create(ctypes.byref(c), ctypes.c_void_p(base), sb, ctypes.c_void_p(base), wb,
                           ctypes.byref(h))
    assert code in (L.OKLS_ERR_NO_DEVICE, L.OKLS_ERR_CUDA)
    assert not h.value


def test_method_is_validated_and_sizes_the_workspace(lib):
    """Shampoo mode drops the N^ and X_a^T binary16 buffers and adds one fp32
    square root per factor (all sizes here are multiples of the 256-byte
    alignment, so the difference is exact)."""
    c = L.config_default(2, 96, 40)
    c.method = 4
    assert lib.okls_state_bytes(ctypes.byref(c), None, None) == L.OKLS_ERR_INVALID_ARG
    c.method = L.METHOD_OKLS
    s0, w0 = L.state_bytes(c)
    c.method = L.METHOD_SHAMPOO
    s1, w1 = L.state_bytes(c)
    B, m, n = 2, 96, 40
    assert s1 == s0
    assert w1 - w0 == 4 * B * (m * m + n * n) - 2 * B * (m * n + n * m)


def test_soap_shapes_and_state(lib):
    """SOAP keeps M, L, R, Q_L, Q_R and V in the state and needs no binary16
    workspace; this build takes m, n <= 16384 (one CTA per matrix up to 128)."""
    c = L.config_default(3, 128, 64)
    c.method = L.METHOD_SOAP
    s, w = L.state_bytes(c)
    assert s >= 4 * 3 * (2 * 128 * 64 + 2 * 128 * 128 + 2 * 64 * 64)
    assert w < 1 << 20
    c.m = 16385
    assert lib.okls_state_bytes(ctypes.byref(c), None, None) == L.OKLS_ERR_UNSUPPORTED
    c.m = 16384
    assert lib.okls_state_bytes(ctypes.byref(c), None, None) == L.OKLS_OK
    # past 128 the batched-GEMM path adds its workspace
    c.m = 300
    s2, w2 = L.state_bytes(c)
    assert w2 >= 4 * 3 * (3 * 300 * 64 + 4 * 300 * 300 + 300 * 300)


def test_soap_batched_path_workspace(lib):
    """The SOAP batched path's workspace is what the header documents: per
    matrix three m x n and one max(mn, m^2, n^2) fp32 buffers, and per side
    d three d x d buffers; up to d = 544 one more and, for d > 128, an
    eigensolver slice of A (full, dp x dp with dp = d rounded up to even), V
    (d x d) and one sweep's rotation log ((dp - 1) x dp floats); past 544 the
    blocked Jacobi slice (four kp x kp buffers, kp = d rounded up to 128, the
    pair rotations and small per-position arrays).  The fixed part
    (descriptor table, scalars, status word, alignment) stays under 1 MiB."""
    def r4(x):
        return (x + 3) // 4 * 4

    def eig(d):
        dp = d + (d & 1)
        return r4(dp * dp) + r4(d * d) + r4((dp - 1) * dp) + 4

    def blocked(d):
        # A and A P, the basis panels (two), pair rotations (128 x 128 each),
        # flags and per-position arrays, the stopping rule's partials
        kp = (d + 127) // 128 * 128
        # (the rotations also as the tensor core's bf16 images: 96 KB per pair)
        return 4 * kp * kp + (kp // 128) * (128 * 128 + 24576) + r4(kp // 128) + 4 * r4(kp) + 4 * 32 + 4

    for B, m, n in [(2, 544, 331), (3, 300, 100), (1, 129, 544), (2, 600, 100), (1, 2048, 5504), (1, 545, 700)]:
        c = L.config_default(B, m, n)
        c.method = L.METHOD_SOAP
        _s, w = L.state_bytes(c)
        floats = B * (3 * m * n + max(m * n, m * m, n * n))
        for d in (m, n):
            floats += B * 3 * d * d
            if d > 544:
                floats += B * blocked(d)
            else:
                floats += B * d * d + (B * eig(d) if d > 128 else 0)
        assert 4 * floats <= w <= 4 * floats + (1 << 20), (B, m, n, w, 4 * floats)


def test_clean_shapes_and_validation(lib):
    """Clean keeps rank-r bases, their eigenvalues and the four blocks'
    moments (linear in m and n); this build takes m, n <= 16384 and
    rank + oversample <= 544, and the rank fields belong to Clean alone."""
    B, m, n, r = 3, 128, 96, 16
    c = L.config_default(B, m, n)
    c.method = L.METHOD_CLEAN
    assert lib.okls_state_bytes(ctypes.byref(c), None, None) == L.OKLS_ERR_INVALID_ARG  # rank 0
    c.rank, c.oversample, c.power_iters = r, 8, 1
    s, w = L.state_bytes(c)
    floats = B * (m * r + n * r + 2 * r + 2 * r * r + m * r + r * n + 2 * r + 1)
    assert 4 * floats <= s <= 4 * floats + 11 * 256
    assert w <= 256 + 4 * B * (m * r + n * r + 2 * r) + 5 * 256
    for field, value, code in [("rank", 0, L.OKLS_ERR_INVALID_ARG), ("oversample", -1, L.OKLS_ERR_INVALID_ARG),
                               ("power_iters", 17, L.OKLS_ERR_INVALID_ARG),
                               ("rank", 89, L.OKLS_ERR_INVALID_ARG),       # r + p > min(m, n)
                               ("m", 16385, L.OKLS_ERR_UNSUPPORTED)]:
        c2 = L.okls_config.from_buffer_copy(c)
        setattr(c2, field, value)
        assert lib.okls_state_bytes(ctypes.byref(c2), None, None) == code, (field, value)
    # past one CTA's shared memory (m > 128 or r + p > 64) the batched-GEMM
    # path takes over: the same state, a workspace of d x (r + p) panels and
    # one m x n fp32 buffer per matrix; r + p above 544 is not supported
    cl = L.config_default(2, 300, 200)
    cl.method, cl.rank, cl.oversample, cl.power_iters = L.METHOD_CLEAN, 32, 16, 1
    s2, w2 = L.state_bytes(cl)
    B2, m2, n2, r2, k2 = 2, 300, 200, 32, 48
    assert 4 * B2 * (m2 * r2 + n2 * r2 + 2 * r2 + 2 * r2 * r2 + m2 * r2 + r2 * n2 + 2 * r2 + 1) <= s2
    assert w2 >= 4 * B2 * (4 * m2 * k2 + m2 * n2)
    cl.m = cl.n = 600
    cl.rank, cl.oversample = 537, 8
    assert lib.okls_state_bytes(ctypes.byref(cl), None, None) == L.OKLS_ERR_UNSUPPORTED
    cl.rank = 536
    L.state_bytes(cl)
    c3 = L.config_default(B, m, n)
    c3.rank = 4
    assert lib.okls_state_bytes(ctypes.byref(c3), None, None) == L.OKLS_ERR_INVALID_ARG
