"""Thin ctypes binding of the C ABI in include/jacobi.h.

Argument marshalling only: every step of the solver runs in the CUDA kernels
of libtbjacobi.so. PyTorch supplies device memory and the stream. There is no
CPU fallback: if the library has not been built, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

SYNC, EXACT_TEMPORAL_BLOCKED, BLOCK_ASYNC = 0, 1, 2
CONTROL_HOST, CONTROL_DEVICE, CONTROL_PERSISTENT = 0, 1, 2
OK, ERR_INVALID_ARG, ERR_CUDA, ERR_NOT_CONVERGED, ERR_NONFINITE, \
    ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5

STRATEGIES = {"sync": SYNC, "etb": EXACT_TEMPORAL_BLOCKED,
              "exact_temporal_blocked": EXACT_TEMPORAL_BLOCKED,
              "ba": BLOCK_ASYNC, "block_async": BLOCK_ASYNC}
CONTROLS = {"host": CONTROL_HOST, "device": CONTROL_DEVICE,
            "persistent": CONTROL_PERSISTENT}
DIVISION_AUTO, DIVISION_IEEE = 0, 1
DIVISIONS = {"auto": DIVISION_AUTO, "ieee": DIVISION_IEEE}
RHS_FUSED, RHS_UNFUSED = 0, 1
RHS_MODES = {"fused": RHS_FUSED, "unfused": RHS_UNFUSED}
ADAPT_NONE, ADAPT_G_ASC, ADAPT_G_DESC, ADAPT_G_FB = 0, 1, 2, 3
ADAPTS = {"none": ADAPT_NONE, "g_asc": ADAPT_G_ASC, "g_desc": ADAPT_G_DESC,
          "g_fb": ADAPT_G_FB}


class Config(ctypes.Structure):
    _fields_ = [("strategy", ctypes.c_int), ("depth", ctypes.c_int),
                ("tile_x", ctypes.c_int), ("tile_y", ctypes.c_int),
                ("check_every", ctypes.c_int), ("tol", ctypes.c_double),
                ("max_sweeps", ctypes.c_longlong), ("control", ctypes.c_int),
                ("division", ctypes.c_int), ("rhs", ctypes.c_int),
                ("adapt", ctypes.c_int), ("overlap_x", ctypes.c_int),
                ("overlap_y", ctypes.c_int)]


class CheckRecord(ctypes.Structure):
    _fields_ = [("depth", ctypes.c_int), ("pad", ctypes.c_int),
                ("sweeps", ctypes.c_longlong), ("rmax", ctypes.c_float),
                ("bmax", ctypes.c_float), ("ms", ctypes.c_float),
                ("pad2", ctypes.c_float)]


class AdaptState(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int), ("depth", ctypes.c_int),
                ("depth_max", ctypes.c_int), ("level", ctypes.c_int),
                ("settle", ctypes.c_int), ("have_prev", ctypes.c_int),
                ("have_ref", ctypes.c_int), ("changes", ctypes.c_int),
                ("rho_prev", ctypes.c_double), ("rate_ref", ctypes.c_double)]


class JacobiError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


_libs = {}
_lock = threading.Lock()


def library_path(checked: bool = False) -> str:
    return _build.LIB_CHECKED if checked else _build.LIB


def load(checked: bool = False):
    """Load libtbjacobi.so, or with checked=True its bounds-checked variant
    libtbjacobi_checked.so (built by __graft_entry__.build() or
    temporal_blocked_jacobi_gb300._build.build_all())."""
    with _lock:
        if checked in _libs:
            return _libs[checked]
        path = library_path(checked)
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, ll, i, f = ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_float
        cfgp = ctypes.POINTER(Config)
        sig = {
            "jacobi_config_default": (i, [cfgp]),
            "jacobi_create": (i, [ctypes.POINTER(vp), i, ll, f, cfgp, vp, vp, vp, vp]),
            "jacobi_rhs": (i, [vp, vp]),
            "jacobi_solve_step": (ll, [vp]),
            "jacobi_sweeps": (ll, [vp, ll]),
            "jacobi_residual": (i, [vp, ctypes.POINTER(f), ctypes.POINTER(f)]),
            "jacobi_set_strategy": (i, [vp, cfgp]),
            "jacobi_run": (ll, [vp, vp, i, ctypes.POINTER(ll)]),
            "jacobi_launch_count": (ll, [vp]),
            "jacobi_division_mode": (i, [vp]),
            "jacobi_destroy": (None, [vp]),
            "jacobi_last_error": (ctypes.c_char_p, [vp]),
            "jacobi_status_string": (ctypes.c_char_p, [i]),
            "jacobi_residual_noalloc": (i, [i, ll, f, vp, vp, vp, vp]),
            "jacobi_check_trace": (ll, [vp, ctypes.POINTER(CheckRecord), ll]),
            "jacobi_adapt_init": (i, [ctypes.POINTER(AdaptState), i, i]),
            "jacobi_adapt_next": (i, [ctypes.POINTER(AdaptState), ctypes.c_double,
                                      ctypes.c_double]),
            "jacobi_tile": (i, [vp, ctypes.POINTER(i), ctypes.POINTER(i)]),
            "jacobi_run_host": (ll, [vp, i, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                     ctypes.POINTER(vp), i, ctypes.POINTER(ll)]),
            "jacobi_bounds_checked": (i, []),
            "jacobi_bounds_selftest": (i, [vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _libs[checked] = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().jacobi_status_string(int(status)).decode()
    except Exception:
        return f"status {status}"


def residual_noalloc(u, b, r, norms, stream=None) -> int:
    """jacobi_residual_noalloc: residual norms of any (u, b) pair into the
    device tensor `norms` (2 floats: rmax, bmax) without allocating anything;
    asynchronous on `stream` (default: the current torch stream of u's
    device). The call is made with u's device current, so u, b, norms and the
    stream must all be on that device.

    Raises ValueError when the tensors are not usable (wrong dtype, shape,
    layout or device); otherwise returns the library's status code (0 on
    success) instead of raising, so a caller inside stream capture can test
    it without unwinding."""
    import torch
    _check_field(u)
    _check_field(b, u.shape)
    if not (isinstance(norms, torch.Tensor) and norms.is_cuda
            and norms.dtype == torch.float32 and norms.numel() >= 2
            and norms.is_contiguous()):
        raise ValueError("norms must be a contiguous float32 CUDA tensor of 2 elements")
    if b.device != u.device or norms.device != u.device:
        raise ValueError("u, b and norms must be on the same device")
    stream = torch.cuda.current_stream(u.device) if stream is None else stream
    if stream.device != u.device:
        raise ValueError("the stream must belong to u's device")
    with torch.cuda.device(u.device):
        return int(load().jacobi_residual_noalloc(
            int(u.shape[0]), int(u.shape[1]), float(r), _ptr(u), _ptr(b),
            _ptr(norms), ctypes.c_void_p(stream.cuda_stream)))


def adapt_depths(policy, depth_max, rhos, mss):
    """Run the library's depth controller (jacobi_adapt_init / _next; host
    code, no GPU) over one time step's checks: returns the D it picks after
    each (rho, ms) pair, starting from [initial D]."""
    st = AdaptState()
    lib = load()
    p = ADAPTS[policy] if isinstance(policy, str) else int(policy)
    rc = lib.jacobi_adapt_init(ctypes.byref(st), p, int(depth_max))
    if rc != OK:
        raise JacobiError(rc, "jacobi_adapt_init")
    out = [st.depth]
    for rho, ms in zip(rhos, mss):
        d = lib.jacobi_adapt_next(ctypes.byref(st), float(rho), float(ms))
        if d < 0:
            raise JacobiError(d, "jacobi_adapt_next")
        out.append(int(d))
    return out


def make_config(strategy="sync", depth=1, tile=(0, 0), check_every=8,
                tol=1e-5, max_sweeps=1 << 22, control="host",
                division="auto", rhs="fused", adapt="none",
                overlap=(0, 0)) -> Config:
    c = Config()
    load().jacobi_config_default(ctypes.byref(c))
    c.strategy = STRATEGIES[strategy] if isinstance(strategy, str) else int(strategy)
    c.depth = int(depth)
    c.tile_x, c.tile_y = int(tile[0]), int(tile[1])
    c.check_every = int(check_every)
    c.tol = float(tol)
    c.max_sweeps = int(max_sweeps)
    c.control = CONTROLS[control] if isinstance(control, str) else int(control)
    c.division = DIVISIONS[division] if isinstance(division, str) else int(division)
    c.rhs = RHS_MODES[rhs] if isinstance(rhs, str) else int(rhs)
    c.adapt = ADAPTS[adapt] if isinstance(adapt, str) else int(adapt)
    c.overlap_x, c.overlap_y = int(overlap[0]), int(overlap[1])
    return c


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check_field(t, shape=None):
    import torch
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32
            and t.dim() == 2 and t.is_contiguous()):
        raise ValueError("fields must be contiguous 2-D float32 CUDA tensors")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"field shape {tuple(t.shape)} != {tuple(shape)}")


def allocate(n: int, ld: int | None = None, device="cuda"):
    """Three zeroed (n, ld) float32 device fields for u, u_alt and b."""
    import torch
    ld = (n + 3) // 4 * 4 if ld is None else ld
    return tuple(torch.zeros((n, ld), dtype=torch.float32, device=device)
                 for _ in range(3))


class Solver:
    """One solver handle over caller-owned fields u, u_alt, b of shape (N, ld).

    u holds uⁿ with its Dirichlet ring on entry; each solved step leaves the
    new iterate in u. All work is enqueued on `stream` (default: the current
    torch stream)."""

    def __init__(self, u, u_alt, b, r, *, strategy="sync", depth=1,
                 tile=(0, 0), check_every=8, tol=1e-5, max_sweeps=1 << 22,
                 control="host", division="auto", rhs="fused", adapt="none",
                 overlap=(0, 0), stream=None, checked=False):
        import torch
        lib = load(checked)
        self._lib = lib
        for t in (u, u_alt, b):
            _check_field(t, u.shape)
        self.n, self.ld = int(u.shape[0]), int(u.shape[1])
        self.u, self.u_alt, self.b = u, u_alt, b
        self.stream = torch.cuda.current_stream(u.device) if stream is None else stream
        self._h = ctypes.c_void_p()
        cfg = make_config(strategy, depth, tile, check_every, tol, max_sweeps,
                          control, division, rhs, adapt, overlap)
        with torch.cuda.device(u.device):
            rc = lib.jacobi_create(ctypes.byref(self._h), self.n, self.ld,
                                   float(r), ctypes.byref(cfg), _ptr(u),
                                   _ptr(u_alt), _ptr(b),
                                   ctypes.c_void_p(self.stream.cuda_stream))
        if rc != OK:
            raise JacobiError(rc, lib.jacobi_last_error(None).decode())
        self.r = float(r)
        self.config = cfg

    # -- helpers -----------------------------------------------------------
    def _raise(self, status):
        raise JacobiError(int(status), self._lib.jacobi_last_error(self._h).decode())

    def _ok(self, rc):
        if rc < 0:
            self._raise(rc)
        return rc

    @property
    def handle(self):
        if not self._h:
            raise RuntimeError("solver is closed")
        return self._h

    # -- C ABI ---------------------------------------------------------------
    def rhs(self, g):
        _check_field(g, self.u.shape)
        self._ok(self._lib.jacobi_rhs(self.handle, _ptr(g)))

    def solve_step(self, raise_on_error=True) -> int:
        k = self._lib.jacobi_solve_step(self.handle)
        return self._ok(k) if raise_on_error else k

    def sweeps(self, launches: int) -> int:
        return self._ok(self._lib.jacobi_sweeps(self.handle, int(launches)))

    def residual(self):
        rm, bm = ctypes.c_float(), ctypes.c_float()
        self._ok(self._lib.jacobi_residual(self.handle, ctypes.byref(rm), ctypes.byref(bm)))
        return rm.value, bm.value

    def bounds_selftest(self) -> int:
        """jacobi_bounds_selftest (bounds-checked library only): the mask of
        the checker's five test accesses that it refused (0x7 when it
        works)."""
        return self._ok(self._lib.jacobi_bounds_selftest(self.handle))

    def set_strategy(self, strategy="sync", depth=1, tile=(0, 0),
                     check_every=8, tol=1e-5, max_sweeps=1 << 22, control="host",
                     division="auto", rhs="fused", adapt="none", overlap=(0, 0)):
        cfg = make_config(strategy, depth, tile, check_every, tol, max_sweeps,
                          control, division, rhs, adapt, overlap)
        self._ok(self._lib.jacobi_set_strategy(self.handle, ctypes.byref(cfg)))
        self.config = cfg

    def run(self, g, steps=10):
        """`steps` backward-Euler steps; returns the list of sweeps per step."""
        _check_field(g, self.u.shape)
        counts = (ctypes.c_longlong * max(steps, 1))()
        total = self._lib.jacobi_run(self.handle, _ptr(g), int(steps), counts)
        if total < 0:
            self._raise(total)
        return [int(counts[s]) for s in range(steps)]

    def run_host(self, u0s, gs, outs, steps=10):
        """jacobi_run_host: independent problems on host tensors (pinned CPU
        float32 tensors of shape (N, ld)); problem i starts from u0s[i] with
        source gs[i] and leaves its final field in outs[i]. The copies
        overlap the solves. Returns the sweeps of every step, per problem."""
        import torch
        count = len(u0s)
        if not (count == len(gs) == len(outs)) or count < 1:
            raise ValueError("u0s, gs and outs must be non-empty and of one length")
        for t in (*u0s, *gs, *outs):
            if not (isinstance(t, torch.Tensor) and not t.is_cuda
                    and t.dtype == torch.float32 and t.is_contiguous()
                    and tuple(t.shape) == (self.n, self.ld)):
                raise ValueError("host buffers must be contiguous float32 CPU "
                                 f"tensors of shape {(self.n, self.ld)}")
        arr = ctypes.c_void_p * count
        pu = arr(*[t.data_ptr() for t in u0s])
        pg = arr(*[t.data_ptr() for t in gs])
        po = arr(*[t.data_ptr() for t in outs])
        counts = (ctypes.c_longlong * (count * steps))()
        total = self._lib.jacobi_run_host(self.handle, count, pu, pg, po, int(steps),
                                          counts)
        if total < 0:
            self._raise(total)
        return [[int(counts[i * steps + s]) for s in range(steps)] for i in range(count)]

    def check_trace(self):
        """The last solve_step's checks: list of dicts (depth, sweeps, rmax,
        bmax, ms); empty under device control."""
        lib = self._lib
        n = lib.jacobi_check_trace(self.handle, None, 0)
        if n < 0:
            self._raise(n)
        recs = (CheckRecord * max(int(n), 1))()
        lib.jacobi_check_trace(self.handle, recs, int(n))
        return [dict(depth=recs[i].depth, sweeps=recs[i].sweeps, rmax=recs[i].rmax,
                     bmax=recs[i].bmax, ms=recs[i].ms) for i in range(int(n))]

    @property
    def division_mode(self) -> int:
        """1 if the kernels use the verified fixed-divisor division, 0 if IEEE."""
        return int(self._ok(self._lib.jacobi_division_mode(self.handle)))

    @property
    def tile(self):
        """(tile_x, tile_y) of the handle's tiled kernel, the default
        resolved; (0, 0) for SYNC; tile_y = 0 is the column-streamed
        exact-temporal-blocking kernel."""
        tx, ty = ctypes.c_int(), ctypes.c_int()
        self._ok(self._lib.jacobi_tile(self.handle, ctypes.byref(tx), ctypes.byref(ty)))
        return tx.value, ty.value

    @property
    def launch_count(self) -> int:
        return int(self._lib.jacobi_launch_count(self.handle))

    @property
    def last_error(self) -> str:
        return self._lib.jacobi_last_error(self.handle).decode()

    def close(self):
        if self._h:
            self._lib.jacobi_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
