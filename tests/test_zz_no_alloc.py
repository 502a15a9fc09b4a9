"""okls_inv_root_noalloc: the inverse root for callers that cannot allocate
device memory (allocators that must not re-enter themselves, fixed device
pools).  Its scratch is a static array in the library; the result must match
okls_inv_root, which takes a caller workspace, two calls in a row must not
see each other's leftovers, and a call must leave the device's free memory
unchanged.

Collected last on purpose: a failure here leaves every other test already
run."""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import spd
from kronecker_factored_second_gb300 import _lib as L

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L.lib()
    torch.cuda.set_device(0)


def _with_workspace(S: torch.Tensor, split: int) -> torch.Tensor:
    lib = L.lib()
    count, d, _ = S.shape
    need = ctypes.c_size_t()
    L.check(lib.okls_inv_root_workspace_bytes(d, count, 10, split, ctypes.byref(need)))
    ws = torch.empty(need.value, dtype=torch.uint8, device="cuda")
    P = torch.empty_like(S)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L.check(lib.okls_inv_root(ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(P.data_ptr()), None, None, d,
                              count, 10, split, 1e-3, 0.0, ctypes.c_void_p(ws.data_ptr()), need.value, st))
    return P


def _no_alloc_into(S: torch.Tensor, P: torch.Tensor, split: int) -> int:
    lib = L.lib()
    count, d, _ = S.shape
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.okls_inv_root_noalloc(ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(P.data_ptr()), d, count,
                                     10, split, 1e-3, 0.0, st)


def _no_alloc(S: torch.Tensor, split: int) -> torch.Tensor:
    P = torch.full_like(S, float("nan"))
    L.check(_no_alloc_into(S, P, split))
    return P


def _fits(d: int, count: int, split: int) -> bool:
    lib = L.lib()
    need = ctypes.c_size_t()
    L.check(lib.okls_inv_root_workspace_bytes(d, count, 10, split, ctypes.byref(need)))
    return need.value <= lib.okls_inv_root_noalloc_capacity()


@pytest.mark.parametrize("d,count,split", [(256, 3, 0), (520, 2, 0), (384, 2, 3), (1024, 2, 0), (1024, 1, 3)])
def test_no_alloc_matches_workspace_entry_twice(d, count, split):
    """Two calls in a row with different inputs: each must match the
    workspace entry point (and the exact root) within the tests' 1e-3 /
    1e-2 bars; identical kernels make them agree far more closely.  The
    1024 cases are the largest requests that fit the static scratch."""
    assert _fits(d, count, split)
    for seed in (1, 2):
        S = torch.tensor(np.stack([spd(d, 100.0, 1000 * seed + 10 * d + i) for i in range(count)]),
                         dtype=torch.float32, device="cuda")
        ref = _with_workspace(S, split).double().cpu().numpy()
        got = _no_alloc(S, split).double().cpu().numpy()
        S64 = S.double().cpu().numpy()
        for b in range(count):
            assert np.all(np.isfinite(got[b]))
            assert O.rel_fro(got[b], ref[b]) < 1e-3
            assert O.rel_fro(got[b], O.inv_root_exact(S64[b])) < 1e-2


def test_no_alloc_leaves_device_memory_unchanged():
    """After a first call on the device (module loading, the scratch's
    address), further calls allocate nothing: the device's free memory and
    torch's allocated bytes are the same before and after each call."""
    S = torch.tensor(np.stack([spd(512, 100.0, 77 + i) for i in range(4)]), dtype=torch.float32, device="cuda")
    P = torch.empty_like(S)
    L.check(_no_alloc_into(S, P, 0))
    torch.cuda.synchronize()
    for _ in range(3):
        free0, _total = torch.cuda.mem_get_info()
        alloc0 = torch.cuda.memory_allocated()
        L.check(_no_alloc_into(S, P, 0))
        torch.cuda.synchronize()
        free1, _total = torch.cuda.mem_get_info()
        assert free1 == free0, (free0, free1)
        assert torch.cuda.memory_allocated() == alloc0
    assert torch.isfinite(P).all()


def test_no_alloc_rejects_requests_beyond_its_scratch():
    """Just past the capacity (three 1024^2 matrices in the plain chain, two
    in the split chain) and far past it (one 2048^2): rejected before any
    launch, with the reason in the last error."""
    lib = L.lib()
    assert not _fits(1024, 3, 0) and not _fits(1024, 2, 3) and not _fits(2048, 1, 0)
    S = torch.zeros(1, 8, 8, device="cuda")
    P = torch.zeros_like(S)
    for (d, count, split) in [(1024, 3, 0), (1024, 2, 3), (2048, 1, 0)]:
        code = lib.okls_inv_root_noalloc(ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(P.data_ptr()), d, count,
                                         10, split, 1e-3, 0.0, None)
        assert code == L.OKLS_ERR_UNSUPPORTED
        assert "static scratch" in L.last_error()
