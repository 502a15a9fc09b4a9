"""PyTorch-facing wrappers over the C ABI (device memory and streams only).

`OklsBatch`        one same-shape batch (the README's 3-D (N, m, n) parameter):
                   state and workspace are torch CUDA tensors handed to
                   okls_create; `step` calls okls_step on the current stream.
`inv_root`         the library's Newton-Schulz inverse root of SPD matrices.
`OnlineKLShampoo`  a torch.optim.Optimizer with the README's constructor
                   (lr, beta1, beta2, eps, weight_decay), one OklsBatch per
                   2-D or 3-D parameter.
`Shampoo`          the classic Shampoo step (summed factors, -1/4 roots)
                   over the same kernels (method="shampoo").
`SOAP`             Adam in the factors' eigenbasis (method="soap"; matrices up
                   to 16384 x 16384 in this build).
`Clean`            block-wise Adam in Nystrom low-rank bases (method="clean";
                   matrices up to 16384 x 16384 and rank + oversample <= 544
                   in this build); the sketch's Gaussian draws come from a
                   torch.Generator and are passed to the library as an input.

All arithmetic happens in libokls.so; nothing here computes on the CPU.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib as L

_DT = {torch.float32: L.OKLS_F32, torch.bfloat16: L.OKLS_BF16}


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("okls: tensors must be contiguous CUDA tensors")


class OklsBatch:
    """A batch of `batch` m x n matrices sharing hyperparameters."""

    def __init__(self, batch: int, m: int, n: int, *, param_dtype=torch.float32,
                 grad_dtype=None, lr: float = 0.09434, beta1: float = 0.9684,
                 beta2: float = 0.9482, eps: float = 1e-9, weight_decay: float = 0.0303,
                 ns_iters: int = 10, ns_split_iters: int = 0, ns_lo: float = 1e-3,
                 ridge: float = 1e-3, variance_correction: bool = True,
                 eps_every_update: bool = True, root_every: int = 1, method: str = "okls",
                 rank: int = 0, oversample: int = 0, power_iters: int = 0, device=None):
        lib = L.lib()
        methods = {"okls": L.METHOD_OKLS, "shampoo": L.METHOD_SHAMPOO, "soap": L.METHOD_SOAP,
                   "clean": L.METHOD_CLEAN}
        if method not in methods:
            raise ValueError(f"okls: method must be one of {sorted(methods)}")
        cfg = L.config_default(batch, m, n)
        cfg.param_dtype = _DT[param_dtype]
        cfg.grad_dtype = _DT[grad_dtype or param_dtype]
        cfg.lr_peak = lr
        cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay = beta1, beta2, eps, weight_decay
        cfg.ns_iters, cfg.ns_split_iters, cfg.ns_lo, cfg.ridge = ns_iters, ns_split_iters, ns_lo, ridge
        cfg.variance_correction = int(variance_correction)
        cfg.eps_every_update = int(eps_every_update)
        cfg.root_every = int(root_every)
        cfg.method = methods[method]
        cfg.rank, cfg.oversample, cfg.power_iters = int(rank), int(oversample), int(power_iters)
        self.method = method
        self.rank, self.oversample = int(rank), int(oversample)
        self.root_every = max(1, int(root_every))
        self.cfg = cfg
        self.batch, self.m, self.n = batch, m, n
        self.param_dtype = param_dtype
        self.grad_dtype = grad_dtype or param_dtype
        sb, wb = L.state_bytes(cfg)
        dev = torch.device("cuda") if device is None else torch.device(device)
        with torch.cuda.device(dev):
            self.state = torch.empty(sb, dtype=torch.uint8, device=dev)
            self.workspace = torch.empty(wb, dtype=torch.uint8, device=dev)
            h = ctypes.c_void_p()
            L.check(lib.okls_create(ctypes.byref(cfg), _ptr(self.state), sb, _ptr(self.workspace), wb,
                                    ctypes.byref(h)))
        self._h = h
        self.device = dev
        self.reset()

    # -- lifecycle
    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            L.lib().okls_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, stream=None):
        L.check(L.lib().okls_reset_state(self._h, _stream(stream)))

    # -- the step
    def step(self, W: torch.Tensor, G: torch.Tensor, lr: float, stream=None, noise: torch.Tensor | None = None):
        """One step; `noise` (Clean only, fp32, `noise_shape`) holds the
        sketch's Gaussian draws and is required when `refresh_due`."""
        _require_cuda(W, G, noise)
        shape = (self.batch, self.m, self.n)
        if tuple(W.shape[-2:]) != shape[1:] or W.numel() != G.numel() or W.numel() != self.batch * self.m * self.n:
            raise ValueError(f"okls: expected W, G of shape {shape}")
        if W.dtype != self.param_dtype or G.dtype != self.grad_dtype:
            raise ValueError("okls: dtype mismatch")
        if noise is None:
            L.check(L.lib().okls_step(self._h, _ptr(W), _ptr(G), float(lr), _stream(stream)))
            return
        if noise.dtype != torch.float32 or tuple(noise.shape) != self.noise_shape:
            raise ValueError(f"okls: noise must be fp32 of shape {self.noise_shape}")
        L.check(L.lib().okls_step_noise(self._h, _ptr(W), _ptr(G), float(lr), _ptr(noise), _stream(stream)))

    @property
    def noise_shape(self) -> tuple[int, int, int]:
        """Clean: per matrix Psi_L (m rows) then Psi_R (n rows), rank + oversample columns."""
        return (self.batch, self.m + self.n, self.rank + self.oversample)

    @property
    def refresh_due(self) -> bool:
        """Clean: the next step re-sketches the bases (t = 1, 1+T, ...)."""
        return self.method == "clean" and self.t % self.root_every == 0

    def query_status(self, stream=None) -> int:
        """Synchronise and return (and clear) the device status word; raises
        OklsError for non-finite values or an expired wait."""
        v = ctypes.c_uint32(0)
        code = L.lib().okls_query_status(self._h, _stream(stream), ctypes.byref(v))
        if code not in (L.OKLS_OK,):
            raise L.OklsError(code, L.last_error())
        return v.value

    def status_nothrow(self, stream=None) -> tuple[int, int]:
        v = ctypes.c_uint32(0)
        code = L.lib().okls_query_status(self._h, _stream(stream), ctypes.byref(v))
        return code, v.value

    # -- state
    def _part_shape(self, part: int):
        B, m, n = self.batch, self.m, self.n
        if self.method == "clean":
            r = self.rank
            return {L.STATE_M: (B, r, r), L.STATE_V: (B, r, r), L.STATE_PA: (B, m, r), L.STATE_PB: (B, n, r),
                    L.STATE_SA: (B, r), L.STATE_SB: (B, r), L.STATE_MA: (B, m, r), L.STATE_MB: (B, r, n),
                    L.STATE_VA: (B, r), L.STATE_VB: (B, r), L.STATE_VC: (B,)}[part]
        return {L.STATE_M: (B, m, n), L.STATE_SA: (B, m, m), L.STATE_SB: (B, n, n),
                L.STATE_PA: (B, m, m), L.STATE_PB: (B, n, n), L.STATE_V: (B, m, n)}[part]

    def get_state(self, part: int, stream=None) -> torch.Tensor:
        out = torch.empty(self._part_shape(part), dtype=torch.float32, device=self.device)
        L.check(L.lib().okls_get_state(self._h, part, _ptr(out), _stream(stream)))
        return out

    def set_state(self, part: int, src: torch.Tensor, stream=None):
        src = src.to(device=self.device, dtype=torch.float32).contiguous()
        if tuple(src.shape) != self._part_shape(part):
            raise ValueError("okls: state shape mismatch")
        L.check(L.lib().okls_set_state(self._h, part, _ptr(src), _stream(stream)))
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()

    @property
    def t(self) -> int:
        v = ctypes.c_int64()
        L.check(L.lib().okls_get_step(self._h, ctypes.byref(v)))
        return v.value

    @t.setter
    def t(self, value: int):
        L.check(L.lib().okls_set_step(self._h, int(value)))

    def set_wait_limit(self, cycles: int = 0, unloaded_tile: int = -1):
        """Wait limit of the GEMM launches of later steps (0: the default)
        and the failure-path test hook (a tile whose operands are never
        loaded; -1: none)."""
        L.check(L.lib().okls_set_wait_limit(self._h, int(cycles), int(unloaded_tile)))

    def profile(self, timing: bool = True):
        """Enable event timing of the GEMM launches of later steps."""
        L.check(L.lib().okls_profile_enable(self._h, int(timing)))

    def read_profile(self) -> dict:
        """Launch counts, algorithmic FLOPs and event time since the last
        read (synchronises on the recorded events)."""
        p = L.okls_profile()
        L.check(L.lib().okls_profile_read(self._h, ctypes.byref(p)))
        return {k: getattr(p, k) for k, _ in L.okls_profile._fields_}

    def _parts(self):
        parts = [("M", L.STATE_M), ("Sa", L.STATE_SA), ("Sb", L.STATE_SB), ("Pa", L.STATE_PA), ("Pb", L.STATE_PB)]
        if self.method == "clean":
            return parts + [("V", L.STATE_V), ("MA", L.STATE_MA), ("MB", L.STATE_MB), ("vA", L.STATE_VA),
                            ("vB", L.STATE_VB), ("vC", L.STATE_VC)]
        return parts + [("V", L.STATE_V)] if self.method == "soap" else parts

    def state_dict(self) -> dict:
        return {"t": self.t, **{k: self.get_state(p).cpu() for k, p in self._parts()}}

    def load_state_dict(self, sd: dict):
        for k, p in self._parts():
            self.set_state(p, sd[k])
        self.t = int(sd["t"])


def inv_root(S: torch.Tensor, *, iters: int = 10, split_iters: int = 0, lo: float = 1e-3,
             ridge: float = 0.0, want_root: bool = False, want_trace: bool = False, stream=None):
    """P = S^(-1/2) (and optionally S^(1/2) and the binary16 iterates) of a
    batch of symmetric d x d fp32 CUDA matrices, by the library's chain."""
    _require_cuda(S)
    if S.dtype != torch.float32:
        raise ValueError("okls.inv_root: fp32 input expected")
    Sb = S if S.dim() == 3 else S.unsqueeze(0)
    count, d, d2 = Sb.shape
    if d != d2:
        raise ValueError("okls.inv_root: square matrices expected")
    lib = L.lib()
    need = ctypes.c_size_t()
    L.check(lib.okls_inv_root_workspace_bytes(d, count, iters, split_iters, ctypes.byref(need)))
    ws = torch.empty(need.value, dtype=torch.uint8, device=S.device)
    P = torch.empty_like(Sb)
    root = torch.empty_like(Sb) if want_root else None
    trace = torch.empty((3 * iters + 1, count, d, d), dtype=torch.float16, device=S.device) \
        if want_trace else None
    L.check(lib.okls_inv_root(_ptr(Sb), _ptr(P), _ptr(root), _ptr(trace), d, count, iters, split_iters,
                              float(lo), float(ridge), _ptr(ws), need.value, _stream(stream)))
    if S.dim() == 2:
        P = P[0]
        root = root[0] if root is not None else None
        trace = trace[:, 0] if trace is not None else None
    out = {"P": P}
    if want_root:
        out["root"] = root
    if want_trace:
        out["trace"] = trace
    return out


class OnlineKLShampoo(torch.optim.Optimizer):
    """Online KL Shampoo over 2-D (m, n) and 3-D (N, m, n) CUDA parameters.

    Constructor and defaults follow the README's usage example; lr is also
    lr_peak for the AdamC correction, and a scheduler may change
    group['lr'] afterwards.
    """

    def __init__(self, params, lr: float = 0.09434, beta1: float = 0.9684, beta2: float = 0.9482,
                 eps: float = 1e-9, weight_decay: float = 0.0303, ns_split_iters: int = 0,
                 ridge: float = 1e-3):
        defaults = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay,
                        ns_split_iters=ns_split_iters, ridge=ridge)
        super().__init__(params, defaults)
        for g in self.param_groups:
            g.setdefault("lr_peak", g["lr"])

    @torch.no_grad()
    def step(self, closure=None):
        loss = closure() if closure is not None else None
        for g in self.param_groups:
            for p in g["params"]:
                if p.grad is None:
                    continue
                if p.dim() not in (2, 3):
                    raise ValueError("OnlineKLShampoo takes 2-D or 3-D matrix parameters only")
                st = self.state[p]
                if "okls" not in st:
                    B = 1 if p.dim() == 2 else p.shape[0]
                    m, n = p.shape[-2:]
                    st["okls"] = OklsBatch(B, m, n, param_dtype=p.dtype, grad_dtype=p.grad.dtype,
                                           lr=g["lr_peak"], beta1=g["beta1"], beta2=g["beta2"],
                                           eps=g["eps"], weight_decay=g["weight_decay"],
                                           ns_split_iters=g["ns_split_iters"], ridge=g["ridge"],
                                           device=p.device)
                st["okls"].step(p.data, p.grad.contiguous(), g["lr"])
        return loss


class Shampoo(torch.optim.Optimizer):
    """Classic Shampoo (optim-book "Shampoo" chapter) over 2-D and 3-D CUDA
    parameters: L += G G^T, R += G^T G, W -= lr L^-1/4 G R^-1/4, with the
    roots refreshed every `root_every` steps (the chapter's 20-100)."""

    def __init__(self, params, lr: float = 1e-2, eps: float = 1e-9, weight_decay: float = 0.0,
                 root_every: int = 1, ns_split_iters: int = 0, ridge: float = 1e-3):
        defaults = dict(lr=lr, eps=eps, weight_decay=weight_decay, root_every=root_every,
                        ns_split_iters=ns_split_iters, ridge=ridge)
        super().__init__(params, defaults)
        for g in self.param_groups:
            g.setdefault("lr_peak", g["lr"])

    @torch.no_grad()
    def step(self, closure=None):
        loss = closure() if closure is not None else None
        for g in self.param_groups:
            for p in g["params"]:
                if p.grad is None:
                    continue
                if p.dim() not in (2, 3):
                    raise ValueError("Shampoo takes 2-D or 3-D matrix parameters only")
                st = self.state[p]
                if "okls" not in st:
                    B = 1 if p.dim() == 2 else p.shape[0]
                    m, n = p.shape[-2:]
                    st["okls"] = OklsBatch(B, m, n, param_dtype=p.dtype, grad_dtype=p.grad.dtype,
                                           lr=g["lr_peak"], eps=g["eps"], weight_decay=g["weight_decay"],
                                           ns_split_iters=g["ns_split_iters"], ridge=g["ridge"],
                                           root_every=g["root_every"], method="shampoo", device=p.device)
                st["okls"].step(p.data, p.grad.contiguous(), g["lr"])
        return loss


class SOAP(torch.optim.Optimizer):
    """SOAP (Clean page, Appendix C, Algorithm 4) over 2-D and 3-D CUDA
    parameters with both dimensions <= 16384: Adam run in the eigenbases of
    the factor EMAs L, R, refreshed every `precondition_frequency` steps."""

    def __init__(self, params, lr: float = 3e-3, betas=(0.95, 0.95), eps: float = 1e-8,
                 weight_decay: float = 0.0, precondition_frequency: int = 10):
        defaults = dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay,
                        precondition_frequency=precondition_frequency)
        super().__init__(params, defaults)
        for g in self.param_groups:
            g.setdefault("lr_peak", g["lr"])

    @torch.no_grad()
    def step(self, closure=None):
        loss = closure() if closure is not None else None
        for g in self.param_groups:
            for p in g["params"]:
                if p.grad is None:
                    continue
                if p.dim() not in (2, 3):
                    raise ValueError("SOAP takes 2-D or 3-D matrix parameters only")
                st = self.state[p]
                if "okls" not in st:
                    B = 1 if p.dim() == 2 else p.shape[0]
                    m, n = p.shape[-2:]
                    b1, b2 = g["betas"]
                    st["okls"] = OklsBatch(B, m, n, param_dtype=p.dtype, grad_dtype=p.grad.dtype,
                                           lr=g["lr_peak"], beta1=b1, beta2=b2, eps=g["eps"],
                                           weight_decay=g["weight_decay"],
                                           root_every=g["precondition_frequency"], method="soap",
                                           device=p.device)
                st["okls"].step(p.data, p.grad.contiguous(), g["lr"])
        return loss


class Clean(torch.optim.Optimizer):
    """Clean (Clean page, Algorithm 1) over 2-D and 3-D CUDA parameters (both
    dimensions <= 16384, rank + oversample <= 544 and <= both dimensions):
    block-wise Adam in rank-`rank` Nystrom bases of
    the two Kronecker factors, re-sketched every `precondition_frequency`
    steps with `oversample` extra Gaussian columns and `power_iters`
    subspace iterations.  The Gaussian draws come from `generator` (a CUDA
    torch.Generator; seeded from `seed` when not given)."""

    def __init__(self, params, lr: float = 3e-3, betas=(0.95, 0.95), eps: float = 1e-8,
                 weight_decay: float = 0.0, rank: int = 16, oversample: int = 8, power_iters: int = 1,
                 precondition_frequency: int = 10, generator: torch.Generator | None = None, seed: int = 0):
        defaults = dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay, rank=rank,
                        oversample=oversample, power_iters=power_iters,
                        precondition_frequency=precondition_frequency)
        super().__init__(params, defaults)
        for g in self.param_groups:
            g.setdefault("lr_peak", g["lr"])
        self._gen = generator
        self._seed = seed

    def _generator(self, device) -> torch.Generator:
        if self._gen is None:
            self._gen = torch.Generator(device=device)
            self._gen.manual_seed(self._seed)
        return self._gen

    @torch.no_grad()
    def step(self, closure=None):
        loss = closure() if closure is not None else None
        for g in self.param_groups:
            for p in g["params"]:
                if p.grad is None:
                    continue
                if p.dim() not in (2, 3):
                    raise ValueError("Clean takes 2-D or 3-D matrix parameters only")
                st = self.state[p]
                if "okls" not in st:
                    B = 1 if p.dim() == 2 else p.shape[0]
                    m, n = p.shape[-2:]
                    b1, b2 = g["betas"]
                    st["okls"] = OklsBatch(B, m, n, param_dtype=p.dtype, grad_dtype=p.grad.dtype,
                                           lr=g["lr_peak"], beta1=b1, beta2=b2, eps=g["eps"],
                                           weight_decay=g["weight_decay"],
                                           root_every=g["precondition_frequency"], method="clean",
                                           rank=g["rank"], oversample=g["oversample"],
                                           power_iters=g["power_iters"], device=p.device)
                ob = st["okls"]
                noise = None
                if ob.refresh_due:
                    noise = torch.randn(ob.noise_shape, generator=self._generator(p.device), device=p.device,
                                        dtype=torch.float32)
                ob.step(p.data, p.grad.contiguous(), g["lr"], noise=noise)
        return loss
