"""ctypes binding of libmoe_nvfp4.so (the C ABI in include/moe_nvfp4.h).

Argument marshalling only: every step of the routed-experts computation runs
in the library's sm_103a kernels.  The functions keep the ABI's names and take
torch CUDA tensors where the ABI takes device pointers.  If the library is not
built, or a call fails, a MoeError is raised -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_nvfp4.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE", 3: "MOE_ERR_NOT_FAST_PATH",
                4: "MOE_ERR_MISALIGNED", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_BAD_EXPERT_ID",
                8: "MOE_ERR_RANGE", 9: "MOE_ERR_SCALE", 10: "MOE_ERR_WORKSPACE_BUSY"}
MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_NOT_FAST_PATH, MOE_ERR_MISALIGNED = 1, 2, 3, 4
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_BAD_EXPERT_ID, MOE_ERR_RANGE = 5, 6, 7, 8
MOE_ERR_SCALE, MOE_ERR_WORKSPACE_BUSY = 9, 10

# Every function include/moe_nvfp4.h declares: name -> (restype, argtypes).
_P, _I, _S = C.c_void_p, C.c_int, C.c_size_t


class moe_plan_desc(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("top_k", C.c_int), ("T_max", C.c_int),
                ("gate_q_dev", C.c_void_p), ("up_q_dev", C.c_void_p), ("down_q_dev", C.c_void_p),
                ("gate_s_dev", C.c_void_p), ("up_s_dev", C.c_void_p), ("down_s_dev", C.c_void_p),
                ("gate_ts_dev", C.c_void_p), ("up_ts_dev", C.c_void_p), ("down_ts_dev", C.c_void_p),
                ("device", C.c_int), ("strict", C.c_int), ("pdl", C.c_int), ("kernel", C.c_int),
                ("shared_gate_q_dev", C.c_void_p), ("shared_up_q_dev", C.c_void_p), ("shared_down_q_dev", C.c_void_p),
                ("shared_gate_s_dev", C.c_void_p), ("shared_up_s_dev", C.c_void_p), ("shared_down_s_dev", C.c_void_p),
                ("shared_ts_dev", C.c_void_p), ("e_lo", C.c_int), ("e_hi", C.c_int), ("act_quant", C.c_int)]


MOE_KERNEL_AUTO, MOE_KERNEL_REGISTER, MOE_KERNEL_TENSOR = 0, 1, 2


class moe_stats_t(C.Structure):
    _fields_ = [("decode_launches", C.c_uint64), ("prefill_launches", C.c_uint64), ("null_launches", C.c_uint64),
                ("group_launches", C.c_uint64), ("rejected_calls", C.c_uint64),
                ("tensor_launches", C.c_uint64), ("route_launches", C.c_uint64), ("small_launches", C.c_uint64),
                ("gemv_launches", C.c_uint64),
                ("num_sms", C.c_int),
                ("stages", C.c_int), ("smem_bytes", C.c_int)]


SIGNATURES = {
    "moe_plan_create": (_I, [C.POINTER(moe_plan_desc), C.POINTER(C.c_void_p)]),
    "moe_plan_destroy": (None, [_P]),
    "moe_workspace_bytes": (_S, [_P, _I]),
    "moe_workspace_init": (_I, [_P, _P, _S, _P]),
    "moe_group": (_I, [_P, _P, _I, _P, _P, _P, _P, _P]),
    "moe_decode": (_I, [_P, _P, _P, _P, _P, _I, _P, _P]),
    "moe_decode_static": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "moe_io_bytes": (_S, [_P, _I, C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)]),
    "moe_step_host": (_I, [_P, _P, _P, _P, _P, _I, _P, _P]),
    "moe_prefill": (_I, [_P, _P, _P, _P, _P, _I, _P, _P]),
    "moe_null_step": (_I, [_P, _P, _P, _P, _P, _I, _P, _P]),
    "moe_route": (_I, [_P, _P, _I, _P, _P, _P]),
    "moe_check": (_I, [_P, _P, _P]),
    "moe_debug_poison_workspace": (_I, [_P, _P, _P]),
    "moe_stats": (_I, [_P, C.POINTER(moe_stats_t)]),
    "moe_last_error": (C.c_char_p, []),
    "moe_status_string": (C.c_char_p, [_I]),
    "moe_abi_version": (_I, []),
}
ABI_SYMBOLS = tuple(SIGNATURES)


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load (once) and prototype the library; raises MoeError if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise MoeError(MOE_ERR_CUDA, f"{path} is not built (run __graft_entry__.build()); "
                                         "there is no fallback path")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, load_library().moe_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise MoeError(MOE_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MoeError(MOE_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MoeError(MOE_ERR_INVALID_ARG, f"{name} must be contiguous")


# ----------------------------------------------------------------------------- ABI functions
_SHARED_ARRAYS = ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s")


def moe_plan_create(weights: dict, H: int, I: int, E: int, top_k: int, T_max: int, device: int = -1,
                    strict: bool = False, pdl: bool = False, kernel: int = MOE_KERNEL_AUTO, shared: dict = None,
                    e_range=None, act_quant: bool = False):
    """weights: dict with gate_q/up_q/down_q/gate_s/up_s/down_s (uint8) and
    gate_ts/up_ts/down_ts (float32) CUDA tensors in the ABI layout (with
    e_range = (e_lo, e_hi): the arrays of those experts only).  shared: an
    optional always-on expert, dict of gate_q/up_q/down_q/gate_s/up_s/down_s
    (one expert's arrays) and ts (float32 [3]).  act_quant: x and h quantised
    once to NVFP4 before each projection (tensor-core kernels only)."""
    lib = load_library()
    for n in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s"):
        _need(weights[n], torch.uint8, n)
    for n in ("gate_ts", "up_ts", "down_ts"):
        _need(weights[n], torch.float32, n)
    sp = [None] * 7
    if shared is not None:
        for n in _SHARED_ARRAYS:
            _need(shared[n], torch.uint8, "shared " + n)
        _need(shared["ts"], torch.float32, "shared ts")
        if shared["ts"].numel() != 3:
            raise MoeError(MOE_ERR_INVALID_ARG, "shared ts must hold the gate, up and down tensor scales")
        sp = [shared[n].data_ptr() for n in _SHARED_ARRAYS] + [shared["ts"].data_ptr()]
    e_lo, e_hi = (0, 0) if e_range is None else (int(e_range[0]), int(e_range[1]))
    d = moe_plan_desc(H, I, E, top_k, T_max,
                      *[weights[n].data_ptr() for n in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s",
                                                        "gate_ts", "up_ts", "down_ts")],
                      device, int(strict), int(pdl), int(kernel), *sp, e_lo, e_hi, int(bool(act_quant)))
    out = C.c_void_p()
    _check(lib.moe_plan_create(C.byref(d), C.byref(out)))
    return out


def moe_plan_destroy(plan):
    load_library().moe_plan_destroy(plan)


def moe_workspace_bytes(plan, T: int) -> int:
    return int(load_library().moe_workspace_bytes(plan, T))


def moe_workspace_init(plan, ws, stream=None):
    _check(load_library().moe_workspace_init(plan, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_group(plan, ids, ws, counts, offsets, perm, stream=None):
    _need(ids, torch.int32, "ids")
    _check(load_library().moe_group(plan, _ptr(ids), ids.shape[0], _ptr(ws), _ptr(counts), _ptr(offsets),
                                    _ptr(perm), _stream(stream)))


def _need_step_shapes(x, ids, w, y):
    """x [T, H], ids and w [T, k], y [>= T, H]: the kernels read T*k ids and
    weights and write T rows of y, so the tensors must agree."""
    T = x.shape[0] if x.dim() == 2 else -1
    if (T < 0 or ids.dim() != 2 or ids.shape[0] != T or tuple(w.shape) != tuple(ids.shape) or y.dim() != 2 or
            y.shape[0] < T or y.shape[1] != x.shape[1]):
        raise MoeError(MOE_ERR_INVALID_ARG, f"shapes x {tuple(x.shape)}, ids {tuple(ids.shape)}, w {tuple(w.shape)}, "
                                            f"y {tuple(y.shape)} are not x [T, H], ids and w [T, k], y [T, H]")


def _step(fn, plan, x, ids, w, y, ws, stream):
    _need(x, torch.bfloat16, "x")
    _need(ids, torch.int32, "ids")
    _need(w, torch.float32, "w")
    _need(y, torch.float32, "y")
    _need_step_shapes(x, ids, w, y)
    _check(fn(plan, _ptr(x), _ptr(ids), _ptr(w), _ptr(y), x.shape[0], _ptr(ws), _stream(stream)))


def moe_decode(plan, x, ids, w, y, ws, stream=None):
    _step(load_library().moe_decode, plan, x, ids, w, y, ws, stream)


def moe_decode_static(plan, x, ids, w, y, check: bool = False, stream=None):
    """moe_decode on the library's own per-device scratch (no workspace
    argument, nothing allocated).  check=True synchronises and raises on a
    device-recorded error."""
    _need(x, torch.bfloat16, "x")
    _need(ids, torch.int32, "ids")
    _need(w, torch.float32, "w")
    _need(y, torch.float32, "y")
    _need_step_shapes(x, ids, w, y)
    _check(load_library().moe_decode_static(plan, _ptr(x), _ptr(ids), _ptr(w), _ptr(y), x.shape[0], int(check),
                                            _stream(stream)))


def moe_io_bytes(plan, T: int):
    """(size, off_ids, off_w) of the packed input block of moe_step_host for
    T tokens: x at 0, ids at off_ids, w at off_w; size 0 for an invalid T."""
    oi, ow = C.c_size_t(0), C.c_size_t(0)
    n = load_library().moe_io_bytes(plan, T, C.byref(oi), C.byref(ow))
    return int(n), int(oi.value), int(ow.value)


def _need_host(t, dtype, nbytes, name):
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise MoeError(MOE_ERR_INVALID_ARG, f"{name} must be a contiguous {dtype} host tensor")
    if t.numel() * t.element_size() < nbytes:
        raise MoeError(MOE_ERR_INVALID_ARG, f"{name} holds {t.numel() * t.element_size()} bytes, needs {nbytes}")


def moe_step_host(plan, io_host, io_dev, y_dev, y_host, T: int, ws, stream=None):
    """The step from a packed host block (x, ids, w at the offsets of
    moe_io_bytes) to a host y: one copy in, then the step, which stores y
    straight into y_host when that is pinned (else into y_dev, followed by one
    copy out); all on `stream` and asynchronous.  io_host / y_host are host
    tensors (pinned for asynchronous copies), io_dev / ws CUDA tensors, y_dev a
    CUDA [>= T, H] tensor."""
    n, _, _ = moe_io_bytes(plan, T) if T > 0 else (0, 0, 0)
    _need_host(io_host, torch.uint8, n, "io_host")
    _need(io_dev, torch.uint8, "io_dev")
    _need(y_dev, torch.float32, "y_dev")
    if io_dev.numel() < n:
        raise MoeError(MOE_ERR_INVALID_ARG, f"io_dev holds {io_dev.numel()} bytes, needs {n}")
    if y_dev.dim() != 2:
        raise MoeError(MOE_ERR_INVALID_ARG, "y_dev must be [T, H]")
    ny = T * y_dev.shape[1] * 4
    if y_dev.numel() * 4 < ny:
        raise MoeError(MOE_ERR_INVALID_ARG, f"y_dev holds {y_dev.numel() * 4} bytes, needs {ny}")
    _need_host(y_host, torch.float32, ny, "y_host")
    _check(load_library().moe_step_host(plan, _ptr(io_host), _ptr(io_dev), _ptr(y_dev), _ptr(y_host), T,
                                          _ptr(ws), _stream(stream)))


def moe_prefill(plan, x, ids, w, y, ws, stream=None):
    _step(load_library().moe_prefill, plan, x, ids, w, y, ws, stream)


def moe_null_step(plan, x, ids, w, y, ws, stream=None):
    _step(load_library().moe_null_step, plan, x, ids, w, y, ws, stream)


def moe_route(plan, logits, ids, w, stream=None):
    """Top-k routing: logits float [T, E] -> ids int32 [T, top_k] and softmax
    weights float [T, top_k] on the device (the ids / w a step then takes)."""
    _need(logits, torch.float32, "logits")
    _need(ids, torch.int32, "ids")
    _need(w, torch.float32, "w")
    T = logits.shape[0] if logits.dim() == 2 else -1
    if T < 0 or ids.dim() != 2 or ids.shape[0] != T or tuple(w.shape) != tuple(ids.shape):
        raise MoeError(MOE_ERR_INVALID_ARG, f"shapes logits {tuple(logits.shape)}, ids {tuple(ids.shape)}, "
                                            f"w {tuple(w.shape)} are not logits [T, E], ids and w [T, k]")
    if not (logits.device == ids.device == w.device):
        raise MoeError(MOE_ERR_INVALID_ARG, "logits, ids and w must be on one device")
    _check(load_library().moe_route(plan, _ptr(logits), T, _ptr(ids), _ptr(w), _stream(stream)))


def moe_check(plan, ws, stream=None) -> int:
    """Synchronise and return the device status code (0 = MOE_OK); clears it."""
    return int(load_library().moe_check(plan, _ptr(ws), _stream(stream)))


def moe_debug_poison_workspace(plan, ws, stream=None):
    _check(load_library().moe_debug_poison_workspace(plan, _ptr(ws), _stream(stream)))


def moe_stats(plan) -> dict:
    s = moe_stats_t()
    _check(load_library().moe_stats(plan, C.byref(s)))
    return {f: getattr(s, f) for f, _ in moe_stats_t._fields_}


def moe_last_error() -> str:
    return load_library().moe_last_error().decode(errors="replace")


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_abi_version() -> int:
    return int(load_library().moe_abi_version())


def expert_range(E: int, rank: int, world: int):
    """Experts [e_lo, e_hi) of rank `rank` when `world` ranks split E experts
    into contiguous ranges whose sizes differ by at most one (the first E %
    world ranks take one more).  Each rank's plan then holds those experts'
    arrays only, and the ranks' partial outputs sum to the whole step."""
    if world < 1 or not 0 <= rank < world or E < world:
        raise MoeError(MOE_ERR_INVALID_ARG, f"cannot split {E} experts over {world} ranks (rank {rank})")
    q, r = divmod(E, world)
    lo = rank * q + min(rank, r)
    return lo, lo + q + (1 if rank < r else 0)


# ----------------------------------------------------------------------------- convenience wrapper
class MoePlan:
    """Owns a plan handle and keeps the weight tensors alive."""

    def __init__(self, weights: dict, H: int, I: int, E: int, top_k: int, T_max: int, device=None,
                 strict: bool = False, pdl: bool = False, kernel: int = MOE_KERNEL_AUTO, shared: dict = None,
                 e_range=None, act_quant: bool = False):
        self.weights, self.shared = weights, shared
        self.H, self.I, self.E, self.top_k, self.T_max = H, I, E, top_k, T_max
        dev = weights["gate_q"].device.index if device is None else device
        self.handle = moe_plan_create(weights, H, I, E, top_k, T_max, device=dev, strict=strict, pdl=pdl,
                                      kernel=kernel, shared=shared, e_range=e_range, act_quant=act_quant)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.moe_plan_destroy(h)
            self.handle = None

    def new_workspace(self, stream=None) -> torch.Tensor:
        n = moe_workspace_bytes(self.handle, 1)
        ws = torch.empty(n, dtype=torch.uint8, device=self.weights["gate_q"].device)
        moe_workspace_init(self.handle, ws, stream)
        return ws

    def step(self, x, ids, w, ws, y=None, stream=None, null: bool = False):
        if x.dim() != 2 or x.shape[1] != self.H or ids.dim() != 2 or ids.shape[1] != self.top_k:
            raise MoeError(MOE_ERR_INVALID_ARG, f"x {tuple(x.shape)} and ids {tuple(ids.shape)} are not "
                                                f"[T, {self.H}] and [T, {self.top_k}]")
        if y is None:
            y = torch.empty((x.shape[0], self.H), dtype=torch.float32, device=x.device)
        if null:
            moe_null_step(self.handle, x, ids, w, y, ws, stream)
        elif x.shape[0] <= 24:
            moe_decode(self.handle, x, ids, w, y, ws, stream)
        else:
            moe_prefill(self.handle, x, ids, w, y, ws, stream)
        return y

    def step_host(self, io: "HostIO", ws, stream=None):
        """moe_step_host on a HostIO block: copy io.x / io.ids / io.w in and
        run the step, which stores y into the pinned io.y.  Asynchronous: io.y
        is valid once the stream has been synchronised."""
        lib = load_library()
        _check(lib.moe_step_host(self.handle, io._host_p, io._dev_p, io._ydev_p, io._yhost_p, io.T, _ptr(ws),
                                   _stream(stream)))
        return io.y

    def route(self, logits, stream=None, ids=None, w=None):
        """Top-k routing of logits [T, E] (float32, on the plan's device): (ids, w).
        The kernel reads T*E logits and writes T*top_k ids and weights, so
        caller-supplied ids / w must be exactly [T, top_k].  Temporaries are
        allocated on `stream`, so the caching allocator does not hand their
        memory out again while the routing queued there may still use it."""
        if logits.dim() != 2 or logits.shape[1] != self.E:
            raise MoeError(MOE_ERR_INVALID_ARG, f"logits {tuple(logits.shape)} is not [T, {self.E}]")
        dev = self.weights["gate_q"].device
        if logits.device != dev:
            raise MoeError(MOE_ERR_INVALID_ARG, f"logits are on {logits.device}, the plan on {dev}")
        T = logits.shape[0]
        for name, t in (("ids", ids), ("w", w)):
            if t is not None and (t.dim() != 2 or tuple(t.shape) != (T, self.top_k)):
                raise MoeError(MOE_ERR_INVALID_ARG, f"{name} {tuple(t.shape)} is not [{T}, {self.top_k}]")
        st = torch.cuda.current_stream(dev) if stream is None else stream
        with torch.cuda.stream(st):
            if ids is None:
                ids = torch.empty((T, self.top_k), dtype=torch.int32, device=dev)
            if w is None:
                w = torch.empty((T, self.top_k), dtype=torch.float32, device=dev)
        moe_route(self.handle, logits, ids, w, st)
        return ids, w

    def step_logits(self, x, logits, ws, y=None, stream=None):
        """Routing, then the step, on one stream: no trip through the host.
        The routing's ids / w (and y, if not given) are allocated on that
        stream, so they stay reserved until the work queued there has run."""
        st = torch.cuda.current_stream(x.device) if stream is None else stream
        ids, w = self.route(logits, st)
        if y is None:
            with torch.cuda.stream(st):
                y = torch.empty((x.shape[0], self.H), dtype=torch.float32, device=x.device)
        return self.step(x, ids, w, ws, y=y, stream=st)

    def group(self, ids, ws, stream=None):
        if ids.dim() != 2 or ids.shape[1] != self.top_k:
            raise MoeError(MOE_ERR_INVALID_ARG, f"ids {tuple(ids.shape)} is not [T, {self.top_k}]")
        dev = ids.device
        counts = torch.empty(self.E, dtype=torch.int32, device=dev)
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(ids.numel(), dtype=torch.int32, device=dev)
        moe_group(self.handle, ids, ws, counts, offsets, perm, stream)
        return counts, offsets, perm

    def check(self, ws, stream=None) -> int:
        return moe_check(self.handle, ws, stream)

    def stats(self) -> dict:
        return moe_stats(self.handle)


class HostIO:
    """Pinned host staging for MoePlan.step_host.  `x` (bf16 [T, H]), `ids`
    (int32 [T, top_k]) and `w` (float [T, top_k]) are views of one pinned block
    that a step copies to the device in one piece; the step's kernels store the
    result straight into `y` (float [T, H], pinned).  `y_dev` is the device
    buffer the library falls back to if the device cannot address `y`.  Write the inputs in place; do not rewrite them while
    an earlier step on this block may still be copying (use one block per step
    in flight).  `y_from` shares another HostIO's y buffers."""

    def __init__(self, plan: MoePlan, T: int, y_from: "HostIO" = None):
        n, oi, ow = moe_io_bytes(plan.handle, T)
        if n == 0:
            raise MoeError(MOE_ERR_INVALID_ARG, f"T={T} outside [1, T_max={plan.T_max}]")
        dev = plan.weights["gate_q"].device
        H, k = plan.H, plan.top_k
        self.T, self.nbytes = T, n
        self.host = torch.zeros(n, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(n, dtype=torch.uint8, device=dev)
        self.x = self.host[:T * H * 2].view(torch.bfloat16).view(T, H)
        self.ids = self.host[oi:oi + T * k * 4].view(torch.int32).view(T, k)
        self.w = self.host[ow:ow + T * k * 4].view(torch.float32).view(T, k)
        if y_from is not None:
            if y_from.T < T or y_from.y.shape[1] != H:
                raise MoeError(MOE_ERR_INVALID_ARG, "y_from's y is smaller than this block's")
            self.y, self.y_dev = y_from.y[:T], y_from.y_dev[:T]
        else:
            self.y = torch.zeros((T, H), dtype=torch.float32).pin_memory()
            self.y_dev = torch.empty((T, H), dtype=torch.float32, device=dev)
        self._host_p, self._dev_p = _ptr(self.host), _ptr(self.dev)
        self._ydev_p, self._yhost_p = _ptr(self.y_dev), _ptr(self.y)
