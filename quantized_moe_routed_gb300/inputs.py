"""Seeded synthetic inputs for the routed-experts MoE step over NVFP4 experts.

This module is the input recipe shared by the tests, the benchmark and the
smoke check.  It holds none of the step's arithmetic (no dequantisation, no
GEMV, no SiLU, no combine): it draws hidden states, router outputs and expert
weights, and encodes the weights into the NVFP4 byte layout the library takes.

The serving pages run their routed experts on EXL3 trellis weights, a bitstream
they never define ("dsv4-carve" README, table "What is in the pack"); the V100
page (section 7.1) moves to an NVFP4 checkpoint because NVFP4 expands into FP16
in registers almost for free.  The expert weights here are NVFP4: E2M1 values,
one E4M3 scale per 16 consecutive elements along the reduction axis, and one
FP32 tensor scale per (expert, projection).  The two-level quantiser is:

* tensor scale   s_g = amax(|W|) / (6 * 448)          (1.0 if amax == 0)
* block code     b   = E4M3_RNE_satfinite((amax_blk / 6) / s_g)
* element code   q   = E2M1_RNE_satfinite(w / (dec(b) * s_g)), sign from signbit(w)
                       (magnitude 0 when the divisor is 0)

All arithmetic is fp32 IEEE (torch ops on either device give identical bytes).
E4M3 encoding/decoding uses torch's float8_e4m3fn casts (a library routine).
E2M1 rounding is round-to-nearest-even on the value grid {0,.5,1,1.5,2,3,4,6}:
ties 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4; |v|>6 -> 6.

Byte layouts (row-major, C order):
  gate_q, up_q : uint8 [E, I, H/2]   element c of a row is the low nibble of
  down_q       : uint8 [E, H, I/2]   byte c//2 when c is even, high when odd
  gate_s, up_s : uint8 [E, I, H/16]  E4M3 scale of elements 16b..16b+15
  down_s       : uint8 [E, H, I/16]
  *_ts         : float32 [E]
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

__all__ = [
    "Workload", "WORKLOADS", "quantize_nvfp4", "make_x", "make_x_variant", "make_topk_w",
    "make_topk_ids", "make_router_logits", "make_expert_weights", "make_uneven_expert_weights", "make_shared_weights",
    "expert_slice",
    "make_inputs", "rotate_ids",
    "rotation_delta", "touched_experts", "algorithmic_bytes",
]


@dataclass(frozen=True)
class Workload:
    """One routed-MoE step shape.  routing in {"uniform", "zipf", "classes"}."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    routing: str
    seed: int = 0
    weight_std: float = 0.02

    def replace(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five workloads of the routed-experts step (T <= 24 decode, plus a prefill chunk).
WORKLOADS = {
    "tiny": Workload("tiny", T=1, H=256, I=128, E=8, k=2, routing="uniform"),
    "decode": Workload("decode", T=1, H=4096, I=1024, E=256, k=8, routing="uniform"),
    "spec_verify": Workload("spec_verify", T=16, H=4096, I=1024, E=256, k=8, routing="zipf"),
    "upper_decode": Workload("upper_decode", T=24, H=4096, I=2048, E=256, k=8, routing="classes"),
    "prefill": Workload("prefill", T=512, H=4096, I=2048, E=256, k=8, routing="uniform"),
}

_E4M3_MAX = 448.0
_E2M1_MAX = 6.0


def _np_rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


# ----------------------------------------------------------------------------- quantiser
def quantize_nvfp4(w: torch.Tensor):
    """Encode an fp32 matrix [rows, K] (K % 16 == 0) as NVFP4.

    Returns (q uint8 [rows, K/2], s uint8 [rows, K/16], ts float32 0-d tensor),
    all on w's device.
    """
    if w.dtype != torch.float32 or w.dim() != 2 or w.shape[1] % 16:
        raise ValueError("quantize_nvfp4 wants float32 [rows, K] with K % 16 == 0")
    rows, K = w.shape
    amax = w.abs().amax()
    ts = torch.where(amax > 0, amax / (_E2M1_MAX * _E4M3_MAX), torch.ones_like(amax))
    blk = w.reshape(rows, K // 16, 16)
    bamax = blk.abs().amax(dim=2)
    sb = ((bamax / _E2M1_MAX) / ts).clamp(max=_E4M3_MAX)
    s_code = sb.to(torch.float8_e4m3fn)
    div = s_code.to(torch.float32) * ts                       # fp32 product, then IEEE division
    div3 = div.unsqueeze(2)
    v = torch.where(div3 > 0, blk.abs() / torch.where(div3 > 0, div3, torch.ones_like(div3)),
                    torch.zeros_like(blk))
    v = v.clamp(max=_E2M1_MAX)
    u8 = torch.uint8
    mag = ((v > 0.25).to(u8) + (v >= 0.75).to(u8) + (v > 1.25).to(u8) + (v >= 1.75).to(u8)
           + (v > 2.5).to(u8) + (v >= 3.5).to(u8) + (v > 5.0).to(u8))
    code = mag | (torch.signbit(blk).to(u8) << 3)
    code = code.reshape(rows, K)
    q = code[:, 0::2] | (code[:, 1::2] << 4)
    return q.contiguous(), s_code.view(torch.uint8).contiguous(), ts.to(torch.float32)


# ----------------------------------------------------------------------------- activations
def make_x(wl: Workload) -> torch.Tensor:
    """Hidden states: N(0,1) fp32 rounded to bf16 (RNE), [T, H], CPU."""
    a = _np_rng(wl.seed, 1).standard_normal((wl.T, wl.H), dtype=np.float32)
    return torch.from_numpy(a).to(torch.bfloat16)


def make_x_variant(wl: Workload, scale_log2: int = 0, outliers=(), outlier_log2: int = 8) -> torch.Tensor:
    """The hidden states of make_x times 2^scale_log2, with the listed channels
    (columns) further multiplied by 2^outlier_log2: the range and outlier-channel
    stress inputs.  Powers of two keep every bf16 value exact (while it stays a
    normal bf16 number), so the input's shape and distribution are unchanged."""
    a = make_x(wl).to(torch.float32) * (2.0 ** scale_log2)
    for c in outliers:
        a[:, c] *= 2.0 ** outlier_log2
    return a.to(torch.bfloat16)


def make_topk_w(wl: Workload) -> torch.Tensor:
    """Router weights: softmax over each token's k N(0,1) logits in float64, cast to fp32."""
    z = _np_rng(wl.seed, 2).standard_normal((wl.T, wl.k))
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p = p / p.sum(axis=1, keepdims=True)
    return torch.from_numpy(p.astype(np.float32))


def make_router_logits(wl: Workload) -> torch.Tensor:
    """Router logits for the routing step in front of the path: N(0,1) fp32
    [T, E] from their own seeded stream (4), CPU."""
    a = _np_rng(wl.seed, 4).standard_normal((wl.T, wl.E), dtype=np.float32)
    return torch.from_numpy(a)


def _ids_uniform(rng, T, k, E):
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=k, replace=False)
    return ids


def _ids_zipf(rng, T, k, E, s=1.0):
    """Zipf(s) over expert ranks, k sequential draws without replacement per token;
    rank -> expert id through a seeded permutation so hot experts are not adjacent."""
    rank_to_expert = rng.permutation(E).astype(np.int32)
    p = 1.0 / np.arange(1, E + 1, dtype=np.float64) ** s
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        avail = np.ones(E, bool)
        for j in range(k):
            c = np.cumsum(np.where(avail, p, 0.0))
            u = rng.random() * c[-1]
            r = int(np.searchsorted(c, u, side="right"))
            while r >= E or not avail[r]:          # guard the u == c[-1] edge
                r = (r - 1) % E
            avail[r] = False
            ids[t, j] = rank_to_expert[r]
    return ids


def _ids_classes(rng, T, k, E, per_class=12, classes=(8, 4, 2, 1)):
    """Experts hit exactly R_e in {8,4,2,1} (per_class experts each), the leftover
    slots filled uniformly from the remaining experts, distinct within a token."""
    if per_class * sum(classes) > T * k or per_class * len(classes) > E:
        raise ValueError("class routing does not fit this shape")
    order = rng.permutation(E).astype(np.int32)
    chosen = [[] for _ in range(T)]
    pos = 0
    for R in classes:                                   # descending R
        for _ in range(per_class):
            e = int(order[pos]); pos += 1
            cand = [t for t in range(T) if len(chosen[t]) < k and e not in chosen[t]]
            cand.sort(key=lambda t: (-(k - len(chosen[t])), t))
            if len(cand) < R:
                raise ValueError("class routing ran out of free slots")
            for t in cand[:R]:
                chosen[t].append(e)
    fillers = order[pos:]
    for t in range(T):
        while len(chosen[t]) < k:
            e = int(fillers[rng.integers(len(fillers))])
            if e not in chosen[t]:
                chosen[t].append(e)
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        ids[t] = rng.permutation(np.array(chosen[t], np.int32))
    return ids


def make_topk_ids(wl: Workload) -> torch.Tensor:
    """Router expert ids [T, k] int32 (distinct within a token), CPU."""
    rng = _np_rng(wl.seed, 3)
    if wl.routing == "uniform":
        ids = _ids_uniform(rng, wl.T, wl.k, wl.E)
    elif wl.routing == "zipf":
        ids = _ids_zipf(rng, wl.T, wl.k, wl.E)
    elif wl.routing == "classes":
        ids = _ids_classes(rng, wl.T, wl.k, wl.E)
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    return torch.from_numpy(ids)


# ----------------------------------------------------------------------------- weights
def _weight_seed(seed: int, proj: int, e: int) -> int:
    return (seed * 1_000_003 + proj * 65_537 + e * 7 + 12_345) & 0x7FFF_FFFF


def make_expert_weights(wl: Workload, device="cpu", experts=None, fill: str = "random"):
    """NVFP4 expert weights in the library's layout, on `device`.

    Each (projection, expert) matrix is drawn N(0, weight_std) in fp32 from its own
    torch generator seeded by (seed, projection, expert) on `device`, then quantised.
    `experts` restricts generation to a subset; the others get `fill`:
    "random" (uniform random bytes, so a read of the wrong expert is visible)
    or "zero".  Returns a dict of tensors.
    """
    dev = torch.device(device)
    E, H, I = wl.E, wl.H, wl.I
    out = {
        "gate_q": torch.empty((E, I, H // 2), dtype=torch.uint8, device=dev),
        "up_q": torch.empty((E, I, H // 2), dtype=torch.uint8, device=dev),
        "down_q": torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev),
        "gate_s": torch.empty((E, I, H // 16), dtype=torch.uint8, device=dev),
        "up_s": torch.empty((E, I, H // 16), dtype=torch.uint8, device=dev),
        "down_s": torch.empty((E, H, I // 16), dtype=torch.uint8, device=dev),
        "gate_ts": torch.empty((E,), dtype=torch.float32, device=dev),
        "up_ts": torch.empty((E,), dtype=torch.float32, device=dev),
        "down_ts": torch.empty((E,), dtype=torch.float32, device=dev),
    }
    want = set(range(E)) if experts is None else {int(e) for e in experts}
    if len(want) < E:
        if fill == "zero":
            for v in out.values():
                v.zero_()
        else:
            g = torch.Generator(device=dev).manual_seed(_weight_seed(wl.seed, 9, 9))
            for name, v in out.items():
                if v.dtype == torch.uint8:
                    v.copy_(torch.randint(0, 256, v.shape, generator=g, device=dev,
                                          dtype=torch.uint8))
                    if name.endswith("_s"):
                        # block scales stay valid E4M3 codes of a quantiser: no sign
                        # bit, no NaN (0x7F becomes 0x7E)
                        v.bitwise_and_(0x7F)
                        v.sub_((v == 0x7F).to(torch.uint8))
                else:
                    v.fill_(1.0)
    shapes = (("gate", I, H), ("up", I, H), ("down", H, I))
    for e in sorted(want):
        for proj, (name, rows, K) in enumerate(shapes):
            g = torch.Generator(device=dev).manual_seed(_weight_seed(wl.seed, proj, e))
            w = torch.randn((rows, K), generator=g, device=dev, dtype=torch.float32)
            w.mul_(wl.weight_std)
            q, s, ts = quantize_nvfp4(w)
            out[name + "_q"][e].copy_(q)
            out[name + "_s"][e].copy_(s)
            out[name + "_ts"][e] = ts
    return out


def make_uneven_expert_weights(wl: Workload, lo: int, hi: int, gain_exp: int, device="cpu"):
    """Every expert drawn as in make_expert_weights, except that before the
    quantisation the gate rows [lo, hi) are scaled by 2^-gain_exp and the down
    columns [lo, hi) by 2^gain_exp: the h rows [lo, hi) then lie about
    gain_exp binades below the rest of h, yet they carry most of y."""
    dev = torch.device(device)
    E, H, I = wl.E, wl.H, wl.I
    out = {n: [] for n in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s", "gate_ts", "up_ts", "down_ts")}
    for e in range(E):
        for proj, (name, rows, K) in enumerate((("gate", I, H), ("up", I, H), ("down", H, I))):
            g = torch.Generator(device=dev).manual_seed(_weight_seed(wl.seed, proj, e))
            w = torch.randn((rows, K), generator=g, device=dev, dtype=torch.float32)
            w.mul_(wl.weight_std)
            if name == "gate":
                w[lo:hi] *= 2.0 ** -gain_exp
            elif name == "down":
                w[:, lo:hi] *= 2.0 ** gain_exp
            q, sc, ts = quantize_nvfp4(w)
            out[name + "_q"].append(q)
            out[name + "_s"].append(sc)
            out[name + "_ts"].append(ts.reshape(1))
    return {n: torch.cat(v) if n.endswith("_ts") else torch.stack(v) for n, v in out.items()}


def make_inputs(wl: Workload, device="cpu", experts="touched", fill="random"):
    """x, topk_ids, topk_w (CPU) and the expert weights (on `device`).

    experts="touched" generates only the experts the routing uses; "all" every one.
    """
    x = make_x(wl)
    ids = make_topk_ids(wl)
    w = make_topk_w(wl)
    sel = None if experts == "all" else touched_experts(ids, wl.E)
    weights = make_expert_weights(wl, device=device, experts=sel, fill=fill)
    return x, ids, w, weights


# ----------------------------------------------------------------------------- benchmark helpers
def touched_experts(ids: torch.Tensor, E: int):
    a = ids.reshape(-1).tolist()
    return sorted({e for e in a if 0 <= e < E})


def rotate_ids(ids: torch.Tensor, step: int, delta: int, E: int) -> torch.Tensor:
    """Per-step relabelling (id + step*delta) mod E of valid ids; keeps every R_e."""
    r = (ids.to(torch.int64) + step * delta) % E
    return torch.where(ids >= 0, r, ids.to(torch.int64)).to(torch.int32)


def rotation_delta(ids: torch.Tensor, E: int, window: int = 4, start: int = 8) -> int:
    """Smallest delta >= start for which `window` consecutive rotated id sets are
    pairwise disjoint (so a step never re-reads an expert a recent step left in L2).
    Falls back to `start` when no delta achieves it (large expert sets overflow L2
    anyway)."""
    base = {e for e in ids.reshape(-1).tolist() if 0 <= e < E}
    for d in range(start, E):
        sets = [{(e + s * d) % E for e in base} for s in range(window)]
        if all(sets[a].isdisjoint(sets[b]) for a in range(window) for b in range(a + 1, window)):
            return d
    return start


def make_shared_weights(wl: Workload, device="cpu"):
    """One always-on (shared) expert in the same NVFP4 layout as a routed
    expert, drawn like expert index E (its own seeded generators): a dict of
    gate_q/up_q [I, H/2], down_q [H, I/2], gate_s/up_s [I, H/16],
    down_s [H, I/16] (uint8) and ts (float32 [3]: gate, up, down)."""
    dev = torch.device(device)
    H, I = wl.H, wl.I
    out, ts = {}, []
    for proj, (name, rows, K) in enumerate((("gate", I, H), ("up", I, H), ("down", H, I))):
        g = torch.Generator(device=dev).manual_seed(_weight_seed(wl.seed, proj, wl.E))
        w = torch.randn((rows, K), generator=g, device=dev, dtype=torch.float32)
        w.mul_(wl.weight_std)
        q, sc, t = quantize_nvfp4(w)
        out[name + "_q"], out[name + "_s"] = q.contiguous(), sc.contiguous()
        ts.append(float(t))
    out["ts"] = torch.tensor(ts, dtype=torch.float32, device=dev)
    return out


def expert_slice(W: dict, e_lo: int, e_hi: int) -> dict:
    """The arrays of experts e_lo .. e_hi-1 only (what a plan serving that
    expert range holds), as contiguous copies."""
    return {k: v[e_lo:e_hi].contiguous() for k, v in W.items()}


def algorithmic_bytes(wl: Workload, ids: torch.Tensor, shared: bool = False) -> int:
    """Bytes the step must move: each touched expert's E2M1 values, E4M3 scales and
    three fp32 tensor scales, plus x (bf16), ids (int32), weights (fp32) and y (fp32)."""
    n = len(touched_experts(ids, wl.E)) + (1 if shared else 0)
    per_expert = 3 * wl.I * wl.H // 2 + 3 * wl.I * wl.H // 16 + 12
    return n * per_expert + wl.T * wl.H * 2 + wl.T * wl.k * 8 + wl.T * wl.H * 4
