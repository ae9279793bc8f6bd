"""Pins of the CPU oracle against things other than itself (no GPU needed).

* the two number formats against the published code tables (tests/golden) and
  against torch's float8_e4m3fn cast (a library routine);
* g and u against an exact brute force in rational arithmetic (fractions);
* SiLU (.) mul against torch.nn.functional.silu;
* the down projection and the combine against torch float64 matmuls on weights
  dequantised by an independent route (golden E2M1 table + torch fp8 cast);
* the grouping against Python's sorted();
* invariants of the step: zero routing weight, token permutation, power-of-two
  scaling, per-slot linearity, empty / out-of-range slots.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import load_golden
from quantized_moe_routed_gb300.inputs import Workload, make_inputs, quantize_nvfp4

E2M1_GOLDEN = {int(c, 16): float(v) for c, v in load_golden("e2m1_values.txt")}


# ------------------------------------------------------------------ formats
def test_e2m1_table_matches_spec():
    assert len(E2M1_GOLDEN) == 16
    for code, val in E2M1_GOLDEN.items():
        got = oracle.dec_e2m1(code)
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_e4m3_golden_and_library():
    for c, v in load_golden("e4m3_values.txt"):
        got = oracle.dec_e4m3(int(c, 16))
        if v == "nan":
            assert np.isnan(got)
        else:
            assert got == float(v) and np.signbit(got) == np.signbit(float(v)), (c, got, v)
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for code in range(256):
        a, b = oracle.dec_e4m3(code), float(lib[code])
        assert (np.isnan(a) and np.isnan(b)) or (a == b and np.signbit(a) == np.signbit(b)), code


# ------------------------------------------------------------------ independent dequant route
def ref_dequant(q, s, ts):
    """Library route: golden E2M1 table for elements, torch fp8 cast for scales."""
    q = torch.as_tensor(q).to(torch.int64)
    codes = torch.stack([q & 15, q >> 4], dim=-1).reshape(q.shape[0], -1)
    tab = torch.tensor([E2M1_GOLDEN[c] for c in range(16)], dtype=torch.float64)
    vals = tab[codes]
    sc = torch.as_tensor(s).contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    return vals * sc.repeat_interleave(16, dim=1) * float(ts)


def test_dequant_matches_library_route():
    g = torch.Generator().manual_seed(5)
    q = torch.randint(0, 256, (24, 40), generator=g, dtype=torch.int32).to(torch.uint8)
    s = torch.randint(0, 0x7E, (24, 5), generator=g, dtype=torch.int32).to(torch.uint8)
    ts = 0.0123
    a = oracle.dequant(q, s, np.float32(ts))
    b = ref_dequant(q, s, np.float32(ts)).numpy()
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ quantiser round trip
def test_quantizer_grid_roundtrip_exact():
    """Grid values (E2M1 value x E4M3 scale x s_g), each block's amax forced to
    6 * scale, encode to the same codes and dequantise to the same values."""
    rng = np.random.default_rng(3)
    rows, K = 8, 64
    nb = K // 16
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    e4 = torch.arange(0x08, 0x7F, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sg_target = 2.0 ** -12
    # block scales chosen so the global amax is exactly 6*448*sg
    bsc = rng.choice(e4, size=(rows, nb))
    bsc[0, 0] = 448.0
    vals = rng.choice(mags, size=(rows, nb, 16)) * rng.choice([-1.0, 1.0], size=(rows, nb, 16))
    vals[:, :, 0] = 6.0                     # amax of each block is 6 * block scale
    w = (vals * bsc[:, :, None] * sg_target).reshape(rows, K).astype(np.float32)
    q, s, ts = quantize_nvfp4(torch.from_numpy(w))
    assert float(ts) == sg_target
    back = oracle.dequant(q, s, float(ts))
    assert np.array_equal(back, w.astype(np.float64))
    assert np.array_equal(s.view(torch.float8_e4m3fn).to(torch.float64).numpy(), bsc)


def test_quantizer_e2m1_ties_to_even():
    """One block with scale 1 and s_g = 1 (amax 6*448 placed in a second block);
    the midpoints between grid values round to the even code."""
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]   # block amax 6 -> block scale 1
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0]
    row = np.zeros(32, np.float32)
    row[:8] = ties
    row[8:16] = -np.array(ties)
    row[16] = 6.0 * 448.0  # second block: amax 2688 -> s_g = 1, block scale 448
    q, s, ts = quantize_nvfp4(torch.from_numpy(row[None, :]))
    assert float(ts) == 1.0
    back = oracle.dequant(q, s, float(ts))[0]
    assert list(back[:8]) == want
    assert list(back[8:16]) == [-v for v in want]
    assert np.signbit(back[8])          # -0.25 rounds to -0 (sign kept)


# ------------------------------------------------------------------ exact brute force on g, u
def _tiny_weights(H, I, E, seed, ts_vals=None):
    g = torch.Generator().manual_seed(seed)
    W = {}
    for name, rows, K in (("gate", I, H), ("up", I, H), ("down", H, I)):
        W[name + "_q"] = torch.randint(0, 256, (E, rows, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)
        # scales 2^-4 .. 2^4 region, never NaN
        W[name + "_s"] = torch.randint(0x18, 0x58, (E, rows, K // 16), generator=g, dtype=torch.int32).to(torch.uint8)
        W[name + "_ts"] = (torch.rand((E,), generator=g) * 0.5 + 0.01).to(torch.float32)
    return W


def _frac_e4m3(code):
    return Fraction(oracle.dec_e4m3(code))  # exact: a dyadic rational


def test_gate_up_exact_against_fractions():
    H, I, E = 64, 48, 3  # I != H so a transposed operand cannot pass
    W = _tiny_weights(H, I, E, seed=11)
    rng = np.random.default_rng(2)
    x = (rng.integers(-24, 25, size=H) / 16.0).astype(np.float64)  # exact in bf16
    e = 2
    g, u, h, o = oracle.expert_pair(x, e, W)
    for name, got in (("gate", g), ("up", u)):
        q = W[name + "_q"][e].numpy()
        s = W[name + "_s"][e].numpy()
        ts = Fraction(float(W[name + "_ts"][e]))
        for i in range(I):
            acc = Fraction(0)
            for c in range(H):
                byte = int(q[i, c // 2])
                nib = (byte >> 4) if (c & 1) else (byte & 15)
                acc += Fraction(E2M1_GOLDEN[nib]) * _frac_e4m3(int(s[i, c // 16])) * ts * Fraction(x[c])
            assert Fraction(got[i]) == acc, (name, i)


def test_silu_mul_and_down_against_torch():
    H, I, E = 64, 48, 2
    W = _tiny_weights(H, I, E, seed=12)
    x = torch.randn(H, generator=torch.Generator().manual_seed(1), dtype=torch.float64)
    for e in range(E):
        g, u, h, o = oracle.expert_pair(x.numpy(), e, W)
        gt = torch.from_numpy(g)
        ut = torch.from_numpy(u)
        h_ref = torch.nn.functional.silu(gt) * ut
        assert torch.allclose(torch.from_numpy(h), h_ref, rtol=1e-14, atol=1e-300)
        Wd = ref_dequant(W["down_q"][e], W["down_s"][e], float(W["down_ts"][e]))
        o_ref = Wd @ torch.from_numpy(h)
        assert torch.allclose(torch.from_numpy(o), o_ref, rtol=1e-11, atol=1e-12 * float(o_ref.abs().max()))


def test_dense_mlp_special_case():
    """k = 1, w = 1: the step is one dense SwiGLU MLP."""
    wl = Workload("t", T=3, H=64, I=32, E=4, k=1, routing="uniform", seed=4)
    x, ids, w, W = make_inputs(wl, experts="all")
    w = torch.ones_like(w)
    y, bad = oracle.moe_forward(x, ids, w, W)
    assert bad == 0
    for t in range(wl.T):
        e = int(ids[t, 0])
        Wg = ref_dequant(W["gate_q"][e], W["gate_s"][e], float(W["gate_ts"][e]))
        Wu = ref_dequant(W["up_q"][e], W["up_s"][e], float(W["up_ts"][e]))
        Wd = ref_dequant(W["down_q"][e], W["down_s"][e], float(W["down_ts"][e]))
        xt = x[t].to(torch.float64)
        ref = Wd @ (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt))
        assert torch.allclose(torch.from_numpy(y[t]), ref, rtol=1e-10, atol=1e-12 * float(ref.abs().max()))


def test_combine_against_torch():
    wl = Workload("t", T=4, H=64, I=32, E=6, k=3, routing="uniform", seed=8)
    x, ids, w, W = make_inputs(wl, experts="all")
    y, _ = oracle.moe_forward(x, ids, w, W)
    for t in range(wl.T):
        acc = torch.zeros(wl.H, dtype=torch.float64)
        for j in range(wl.k):
            e = int(ids[t, j])
            Wg = ref_dequant(W["gate_q"][e], W["gate_s"][e], float(W["gate_ts"][e]))
            Wu = ref_dequant(W["up_q"][e], W["up_s"][e], float(W["up_ts"][e]))
            Wd = ref_dequant(W["down_q"][e], W["down_s"][e], float(W["down_ts"][e]))
            xt = x[t].to(torch.float64)
            acc += float(w[t, j]) * (Wd @ (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt)))
        assert torch.allclose(torch.from_numpy(y[t]), acc, rtol=1e-10, atol=1e-12 * float(acc.abs().max()))


# ------------------------------------------------------------------ invariants
def make_small_case():
    wl = Workload("t", T=5, H=128, I=64, E=8, k=3, routing="uniform", seed=21)
    return wl, make_inputs(wl, experts="all")


@pytest.fixture(scope="module")
def small_case():
    return make_small_case()


def test_zero_weights_give_zero(small_case):
    wl, (x, ids, w, W) = small_case
    y, _ = oracle.moe_forward(x, ids, torch.zeros_like(w), W)
    assert np.all(y == 0.0)


def test_token_permutation_permutes_output(small_case):
    wl, (x, ids, w, W) = small_case
    y, _ = oracle.moe_forward(x, ids, w, W)
    p = torch.tensor([3, 0, 4, 1, 2])
    y2, _ = oracle.moe_forward(x[p], ids[p], w[p], W)
    assert np.array_equal(y2, y[p.numpy()])


def test_power_of_two_scaling(small_case):
    wl, (x, ids, w, W) = small_case
    y, _ = oracle.moe_forward(x, ids, w, W)
    y2, _ = oracle.moe_forward(x, ids, w * 8.0, W)
    assert np.array_equal(y2, 8.0 * y)


def test_slot_linearity(small_case):
    wl, (x, ids, w, W) = small_case
    y, _ = oracle.moe_forward(x, ids, w, W)
    acc = np.zeros_like(y)
    for j in range(wl.k):
        ids_j = torch.full_like(ids, -1)
        ids_j[:, j] = ids[:, j]
        yj, _ = oracle.moe_forward(x, ids_j, w, W)
        acc += yj
    assert np.allclose(acc, y, rtol=1e-12, atol=1e-13 * np.abs(y).max())


def test_empty_and_bad_slots(small_case):
    wl, (x, ids, w, W) = small_case
    ids2 = ids.clone()
    ids2[1, 0] = -1
    ids2[2, 1] = wl.E + 3
    y, bad = oracle.moe_forward(x, ids2, w, W)
    assert bad == 1
    ref = ids.clone()
    ref[1, 0] = -1
    ref[2, 1] = -1
    y_ref, _ = oracle.moe_forward(x, ref, w, W)
    assert np.array_equal(y, y_ref)
    # a token with no valid slot has y == 0
    ids3 = ids.clone()
    ids3[0, :] = -1
    y3, _ = oracle.moe_forward(x, ids3, w, W)
    assert np.all(y3[0] == 0.0)


def test_duplicate_slots_add(small_case):
    wl, (x, ids, w, W) = small_case
    w = torch.round(w * 256) / 256          # dyadic weights: w0 + w1 is exact in fp32
    ids2 = ids.clone()
    ids2[:, 1] = ids2[:, 0]
    y, _ = oracle.moe_forward(x, ids2, w, W)
    ids_a = ids2.clone()
    ids_a[:, 1] = -1
    w_a = w.clone()
    w_a[:, 0] = w[:, 0] + w[:, 1]
    y_a, _ = oracle.moe_forward(x, ids_a, w_a, W)
    assert np.allclose(y, y_a, rtol=1e-12, atol=1e-13 * np.abs(y).max())


def test_token_subset_matches_full(small_case):
    wl, (x, ids, w, W) = small_case
    y, _ = oracle.moe_forward(x, ids, w, W)
    ys, _ = oracle.moe_forward(x, ids, w, W, tokens=[4, 1])
    assert np.array_equal(ys, y[[4, 1]])


def test_thread_count_does_not_change_result(small_case):
    wl, (x, ids, w, W) = small_case
    a, _ = oracle.moe_forward(x, ids, w, W, n_threads=1)
    b, _ = oracle.moe_forward(x, ids, w, W, n_threads=4)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ grouping
@pytest.mark.parametrize("T,k,E,seed", [(1, 2, 8, 0), (16, 8, 256, 1), (24, 8, 256, 2),
                                        (512, 8, 256, 3), (0, 8, 256, 4), (7, 4, 5, 5)])
def test_group_against_sorted(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-2, E + 2, size=(T, k)).astype(np.int32)
    counts, offsets, perm, bad = oracle.group(ids, E)
    flat = ids.reshape(-1)
    valid = [(int(e), p) for p, e in enumerate(flat) if 0 <= e < E]
    ref = [p for _, p in sorted(valid)]
    assert list(perm[:len(ref)]) == ref
    assert all(v == -1 for v in perm[len(ref):])
    assert bad == int(np.sum(flat >= E))
    for e in range(E):
        assert counts[e] == sum(1 for v in flat if v == e)
    assert offsets[0] == 0 and list(np.diff(offsets)) == list(counts)


# ------------------------------------------------------------------ routing (top-k + softmax in front of the step)
def _route_brute(logits, k):
    """numpy: stable sort by descending logit (NaN as -inf), softmax in float64."""
    lg = np.where(np.isnan(logits), -np.inf, logits.astype(np.float64))
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(lg, order, axis=1)
    z = np.exp(sel - sel[:, :1])
    return order.astype(np.int32), (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("T,E,k,seed", [(1, 256, 8, 0), (16, 256, 8, 1), (5, 7, 7, 2), (3, 1024, 16, 3), (0, 8, 2, 4)])
def test_route_against_brute_force(T, E, k, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.route(logits, k)
    ref_ids, ref_w = _route_brute(logits, k)
    assert np.array_equal(ids, ref_ids)
    assert np.allclose(w, ref_w, rtol=2.5e-7, atol=0)


def test_route_ties_nan_and_extremes():
    lg = np.array([[0.5, 2.0, 2.0, -1.0, np.nan, 3.0],
                   [1.0, 1.0, 1.0, 1.0, 1.0, 1.0],
                   [1000.0, 999.0, -1000.0, 998.0, 0.0, 0.0],
                   [-np.inf] * 6,
                   [np.nan, -5.0, 0.25, np.nan, 0.5, -5.0],
                   [1.0, np.inf, 0.0, np.inf, 5.0, np.inf],
                   [np.inf, -np.inf, 3.0, 2.0, 1.0, 0.0]], np.float32)
    ids, w = oracle.route(lg, 3)
    assert ids.tolist() == [[5, 1, 2], [0, 1, 2], [0, 1, 3], [0, 1, 2], [4, 2, 1], [1, 3, 5], [0, 2, 3]]
    assert np.allclose(w[1], 1 / 3, rtol=1e-7)                     # equal logits, equal weights
    e = np.exp([0.0, -1.0, -2.0])
    assert np.allclose(w[2], e / e.sum(), rtol=2.5e-7)             # large logits: no overflow
    assert np.all(w[3] == 0.0)                                       # nothing finite to weigh
    assert np.allclose(w[5], 1 / 3, rtol=1e-7)                       # +inf winners share the weight
    assert w[6].tolist() == [1.0, 0.0, 0.0]                          # one +inf winner takes it all
    assert np.allclose(w[:3].astype(np.float64).sum(axis=1), 1.0, atol=1e-6)


def test_route_invariants():
    rng = np.random.default_rng(9)
    lg = rng.standard_normal((6, 64)).astype(np.float32)
    ids, w = oracle.route(lg, 8)
    ids2, w2 = oracle.route(lg + np.float32(4.0), 8)                # softmax is shift-invariant
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-6)
    perm = rng.permutation(64)                                       # relabelling experts relabels ids
    ids3, w3 = oracle.route(lg[:, perm], 8)
    assert np.array_equal(perm[ids3], ids) and np.array_equal(w3, w)
    full, wf = oracle.route(lg, 64)                                  # k = E: the whole descending order
    assert np.array_equal(full, np.argsort(-lg, axis=1, kind="stable"))
    assert np.all(np.diff(wf, axis=1) <= 0)
