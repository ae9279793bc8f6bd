"""CPU oracle of the routed-experts MoE step over NVFP4 experts.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library and its binding never do.
It shares no code with the CUDA path.  The arithmetic lives in moe_oracle.c
(plain C, double precision, sums in index order); this module compiles it with
gcc on first use and marshals numpy / torch CPU arrays into it.

Functions:
  dec_e2m1(code), dec_e4m3(code)   -- format definitions (code -> value)
  dequant(q, s, ts)                -- [rows, K] NVFP4 matrix -> float64
  expert_pair(...)                 -- g, u, h, o for one (token, expert) pair
  moe_forward(...)                 -- y (float64) for all or selected tokens
  group(ids, E)                    -- counts, offsets, perm (stable) + bad count
  route(logits, k)                 -- top-k ids and softmax weights per token
  quant_row_nvfp4(v)               -- one row quantised once to NVFP4, dequantised
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/libmoe_oracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P = C.c_void_p
            i = C.c_int
            lib.oracle_dec_e2m1.argtypes = [C.c_uint]
            lib.oracle_dec_e2m1.restype = C.c_double
            lib.oracle_dec_e4m3.argtypes = [C.c_uint]
            lib.oracle_dec_e4m3.restype = C.c_double
            lib.oracle_dequant.argtypes = [P, P, C.c_float, i, i, P]
            lib.oracle_dequant.restype = None
            lib.oracle_expert_pair.argtypes = [i, i, i, P] + [P] * 9 + [P, P, P, P, i]
            lib.oracle_expert_pair.restype = None
            lib.oracle_moe_forward.argtypes = [i, i, i, i, i, P, P, P] + [P] * 9 + [P, i, P, i]
            lib.oracle_moe_forward.restype = C.c_int
            lib.oracle_moe_forward_ext.argtypes = ([i, i, i, i, i, P, P, P] + [P] * 9 + [i, i] + [P] * 7 + [i] +
                                                   [P, i, P, i])
            lib.oracle_moe_forward_ext.restype = C.c_int
            lib.oracle_group.argtypes = [P, i, i, P, P, P]
            lib.oracle_group.restype = C.c_int
            lib.oracle_quant_row.argtypes = [P, i, P]
            lib.oracle_quant_row.restype = None
            lib.oracle_route.argtypes = [P, i, i, i, P, P]
            lib.oracle_route.restype = C.c_int
            _lib = lib
    return _lib


def _np(a, dtype):
    """Contiguous numpy array of `dtype` from a numpy array or a CPU torch tensor
    (bf16 tensors are passed as their uint16 bit patterns)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


def dec_e2m1(code: int) -> float:
    return _load().oracle_dec_e2m1(code)


def dec_e4m3(code: int) -> float:
    return _load().oracle_dec_e4m3(code)


def dequant(q, s, ts) -> np.ndarray:
    """[rows, K/2] packed E2M1 + [rows, K/16] E4M3 + fp32 scalar -> float64 [rows, K]."""
    q = _np(q, np.uint8)
    s = _np(s, np.uint8)
    rows, K = q.shape[0], q.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    _load().oracle_dequant(_p(q), _p(s), C.c_float(float(ts)), rows, K, _p(out))
    return out


def _weights(W):
    names = ("gate_q", "gate_s", "gate_ts", "up_q", "up_s", "up_ts", "down_q", "down_s", "down_ts")
    arrs = []
    for n in names:
        arrs.append(_np(W[n], np.float32 if n.endswith("_ts") else np.uint8))
    return arrs


def expert_pair(x_row, e: int, W, n_threads: int = 0):
    """g, u, h (float64 [I]) and o (float64 [H]) for one token row through expert e.
    x_row: float64-convertible [H] (bf16 tensors convert exactly)."""
    arrs = _weights(W)
    H = arrs[0].shape[2] * 2
    I = arrs[0].shape[1]
    try:
        import torch
        if isinstance(x_row, torch.Tensor):
            x_row = x_row.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    xr = np.ascontiguousarray(x_row, dtype=np.float64)
    g = np.empty(I, np.float64)
    u = np.empty(I, np.float64)
    h = np.empty(I, np.float64)
    o = np.empty(H, np.float64)
    _load().oracle_expert_pair(H, I, int(e), _p(xr), *[_p(a) for a in arrs],
                               _p(g), _p(u), _p(h), _p(o), int(n_threads))
    return g, u, h, o


def moe_forward(x, ids, w, W, tokens=None, n_threads: int = 0, shared=None, e_range=None, E=None,
                act_quant: bool = False):
    """y (float64 [n, H]) for `tokens` (default all) and the count of ids >= E.

    shared: optional dict gate_q/gate_s/up_q/up_s/down_q/down_s (one expert's
    arrays) and ts (float32 [3]: gate, up, down tensor scales) -- an always-on
    expert added to every token with weight 1 after the routed slots.
    e_range: (e_lo, e_hi) -- W holds experts e_lo .. e_hi-1 only; ids outside
    the range are another device's and contribute nothing; E (required with
    e_range) is the total expert count that bounds valid ids.
    act_quant: x and h quantised once to NVFP4 before the projections."""
    arrs = _weights(W)
    El, I, H2 = arrs[0].shape
    H = H2 * 2
    if e_range is None:
        e_lo, e_hi, E = 0, El, El
    else:
        e_lo, e_hi = e_range
        if E is None or e_hi - e_lo != El:
            raise ValueError("e_range needs E and W holding exactly e_hi - e_lo experts")
    sh = [None] * 7
    if shared is not None:
        sh = [_np(shared[n], np.uint8) for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")]
        sh.append(_np(shared["ts"], np.float32))
    xb = _np(x, np.uint16)
    T = xb.shape[0]
    idsa = _np(ids, np.int32)
    k = idsa.shape[1]
    wa = _np(w, np.float32)
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = tok.shape[0]
    y = np.zeros((n, H), np.float64)
    bad = _load().oracle_moe_forward_ext(H, I, E, k, T, _p(xb), _p(idsa), _p(wa),
                                         *[_p(a) for a in arrs], int(e_lo), int(e_hi),
                                         *[None if a is None else _p(a) for a in sh], int(bool(act_quant)),
                                         None if tok is None else _p(tok), n, _p(y), int(n_threads))
    if bad < 0:
        raise ValueError("oracle_moe_forward rejected its arguments")
    return y, bad


def group(ids, E: int):
    """Stable counting sort of flat pairs p = t*k + j by expert: (counts, offsets, perm, bad)."""
    idsa = _np(ids, np.int32).reshape(-1)
    P = idsa.shape[0]
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(max(P, 1), np.int32)
    bad = _load().oracle_group(_p(idsa), P, E, _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm[:P], bad


def quant_row_nvfp4(v) -> np.ndarray:
    """One activation row (fp32, length a multiple of 16) quantised once to
    NVFP4 (row prescale, per-16 E4M3 scale, E2M1) and dequantised (float64)."""
    va = _np(v, np.float32).reshape(-1)
    if va.shape[0] % 16:
        raise ValueError("the row length must be a multiple of 16")
    out = np.empty(va.shape[0], np.float64)
    _load().oracle_quant_row(_p(va), va.shape[0], _p(out))
    return out


def route(logits, k: int):
    """Top-k experts per token by logit (ties: smaller index; NaN as -inf) and
    the softmax of the selected logits: (ids int32 [T, k], w float32 [T, k])."""
    lg = _np(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    if _load().oracle_route(_p(lg), T, E, int(k), _p(ids), _p(w)) != 0:
        raise ValueError("oracle_route rejected its arguments")
    return ids, w
