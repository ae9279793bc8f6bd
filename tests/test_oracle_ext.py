"""Pins of the oracle's three extensions of the step, each against something
other than the oracle's own formula:

* shared expert -- an always-on SwiGLU expert added with weight 1 after the
  routed slots: alone it is the dense MLP (torch float64 matmuls on an
  independent dequantisation), and it adds exactly to the routed part;
* expert range -- a plan serving experts [e_lo, e_hi) (arrays of those only):
  partial outputs over disjoint ranges sum to the whole step, and one expert's
  range equals the whole step with every other slot emptied;
* single NVFP4 activation quantisation -- one row prescale, per-16 E4M3 scale
  (the smallest E4M3 value >= block max / 6), E2M1 round-to-nearest-even:
  exact on grid rows, the tie rule, scale and sign invariance, the error bound.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300.inputs import Workload, expert_slice, make_inputs, make_shared_weights


def ref_dequant(q, s, ts):
    """Independent dequantisation: OCP E2M1 table and torch's float8_e4m3fn cast."""
    e2m1 = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float64)
    q = torch.as_tensor(q).to(torch.int64)
    lo, hi = q & 15, q >> 4
    vals = torch.stack([e2m1[lo], e2m1[hi]], dim=-1).reshape(q.shape[0], -1)
    sc = torch.as_tensor(s).view(torch.float8_e4m3fn).to(torch.float64).repeat_interleave(16, dim=1)
    return vals * sc * float(ts)


def dense(shared, x_row):
    Wg = ref_dequant(shared["gate_q"], shared["gate_s"], shared["ts"][0])
    Wu = ref_dequant(shared["up_q"], shared["up_s"], shared["ts"][1])
    Wd = ref_dequant(shared["down_q"], shared["down_s"], shared["ts"][2])
    xt = x_row.to(torch.float64)
    return Wd @ (torch.nn.functional.silu(Wg @ xt) * (Wu @ xt))


def make_case():
    wl = Workload("ext", T=4, H=128, I=64, E=8, k=3, routing="uniform", seed=51)
    x, ids, w, W = make_inputs(wl, experts="all")
    return wl, x, ids, w, W, make_shared_weights(wl)


@pytest.fixture(scope="module")
def case():
    return make_case()


# ------------------------------------------------------------------ shared expert
def test_shared_expert_alone_is_the_dense_mlp(case):
    wl, x, ids, w, W, S = case
    empty = torch.full_like(ids, -1)
    y, bad = oracle.moe_forward(x, empty, w, W, shared=S)
    assert bad == 0
    for t in range(wl.T):
        ref = dense(S, x[t])
        assert torch.allclose(torch.from_numpy(y[t]), ref, rtol=1e-10, atol=1e-12 * float(ref.abs().max()))


def test_shared_expert_adds_after_the_routed_slots(case):
    wl, x, ids, w, W, S = case
    y_all, _ = oracle.moe_forward(x, ids, w, W, shared=S)
    y_routed, _ = oracle.moe_forward(x, ids, w, W)
    y_shared, _ = oracle.moe_forward(x, torch.full_like(ids, -1), w, W, shared=S)
    assert np.array_equal(y_all, y_routed + y_shared)            # the same double additions, in that order
    y_zero, _ = oracle.moe_forward(x, ids, torch.zeros_like(w), W, shared=S)
    assert np.array_equal(y_zero, y_shared)                      # zero routing weights leave the shared part


def test_shared_expert_zero_weights_change_nothing(case):
    wl, x, ids, w, W, S = case
    Z = {k: torch.zeros_like(v) for k, v in S.items()}
    y_z, _ = oracle.moe_forward(x, ids, w, W, shared=Z)
    y, _ = oracle.moe_forward(x, ids, w, W)
    assert np.array_equal(y_z, y)


# ------------------------------------------------------------------ expert range
@pytest.mark.parametrize("cut", [1, 3, 7])
def test_expert_range_partials_sum_to_the_whole_step(case, cut):
    wl, x, ids, w, W, S = case
    y, bad = oracle.moe_forward(x, ids, w, W, shared=S)
    ya, bad_a = oracle.moe_forward(x, ids, w, expert_slice(W, 0, cut), e_range=(0, cut), E=wl.E, shared=S)
    yb, bad_b = oracle.moe_forward(x, ids, w, expert_slice(W, cut, wl.E), e_range=(cut, wl.E), E=wl.E)
    assert bad == bad_a == bad_b == 0                            # another plan's ids are not errors
    assert np.allclose(ya + yb, y, rtol=1e-12, atol=1e-14 * np.abs(y).max())


def test_one_expert_range_is_the_step_with_other_slots_emptied(case):
    wl, x, ids, w, W, S = case
    e = int(ids[0, 0])
    ye, _ = oracle.moe_forward(x, ids, w, expert_slice(W, e, e + 1), e_range=(e, e + 1), E=wl.E)
    masked = torch.where(ids == e, ids, torch.full_like(ids, -1))
    ym, _ = oracle.moe_forward(x, masked, w, W)
    assert np.array_equal(ye, ym)


def test_expert_range_still_flags_ids_past_E(case):
    wl, x, ids, w, W, S = case
    bad_ids = ids.clone()
    bad_ids[1, 2] = wl.E + 5
    _, bad = oracle.moe_forward(x, bad_ids, w, expert_slice(W, 0, 4), e_range=(0, 4), E=wl.E)
    assert bad == 1


# ------------------------------------------------------------------ single NVFP4 quantisation
E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def test_quant_row_is_exact_on_the_grid():
    rng = np.random.default_rng(3)
    for s_exp in (-3, 0, 5):
        rows = []
        for b in range(8):
            blk = rng.choice(E2M1, 16) * rng.choice([-1, 1], 16)
            blk[rng.integers(16)] = 6.0          # block max 6 s: the scale is exactly s
            rows.append(blk * 2.0 ** (s_exp - b % 3))
        v = np.concatenate(rows).astype(np.float32)
        assert np.array_equal(oracle.quant_row_nvfp4(v), v.astype(np.float64))


def test_quant_row_ties_to_even():
    v = np.array([6, 2.5, 0.75, 5, 1.25, 3.5, -1.75, 0.25, -0.75, 4.5, 0, 1, 2, 3, 4, -6], np.float32)
    q = oracle.quant_row_nvfp4(v)
    assert q.tolist() == [6, 2, 1, 4, 1, 4, -2, 0, -1, 4, 0, 1, 2, 3, 4, -6]


@pytest.mark.parametrize("seed", range(6))
def test_quant_row_scale_sign_invariance_and_bound(seed):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(256) * np.exp(rng.uniform(-2, 2, 256))).astype(np.float32)
    v[rng.integers(256, size=3)] *= 64.0                         # outliers
    q = oracle.quant_row_nvfp4(v)
    for m in (-20, 7, 30):                                       # a power of two moves through exactly
        assert np.array_equal(oracle.quant_row_nvfp4(v * np.float32(2.0 ** m)), q * 2.0 ** m)
    assert np.array_equal(oracle.quant_row_nvfp4(-v), -q)
    blk = np.abs(v.astype(np.float64)).reshape(-1, 16).max(axis=1).repeat(16)
    # s <= (9/8) block max / 6 (E4M3 steps of 1/8 above the ceiling), E2M1 half-gaps <= s
    assert np.all(np.abs(q - v) <= 9.0 / 48.0 * blk * (1 + 1e-6))
    # no element saturates: every quantised magnitude stays within a half-gap of its value
    assert np.all(np.abs(q) <= np.abs(v) + 9.0 / 48.0 * blk * (1 + 1e-6))


def test_quant_row_raises_the_block_scale():
    """A worked example of the rule, by hand: the block [6.375, 1, 0, ...] has
    row prescale 2^8 (6.375 = 1.59375 * 2^2, so 10 - 2), prescaled max 1632,
    1632 / 6 = 272 between the E4M3 values 256 and 288: the scale is raised to
    288 (round-to-nearest-even alone would give 256 and saturate the element
    at 6).  Codes: RNE(1632 / 288 = 5.67) = 6 and RNE(256 / 288 = 0.89) = 1,
    so the values are 6 * 288 / 256 = 6.75 and 288 / 256 = 1.125."""
    v = np.zeros(16, np.float32)
    v[0], v[1] = 6.375, 1.0
    q = oracle.quant_row_nvfp4(v)
    assert q[0] == 6.75 and q[1] == 1.125 and np.all(q[2:] == 0)


def test_quant_row_of_zeros_and_tiny_blocks():
    v = np.zeros(32, np.float32)
    assert np.all(oracle.quant_row_nvfp4(v) == 0)
    v[3] = 1e-30
    v[20] = 1.0
    q = oracle.quant_row_nvfp4(v)
    # a lone 1.0: prescale 2^11, scale = the smallest E4M3 >= 2048 / 6 (352),
    # code RNE(2048 / 352) = 6, so 6 * 352 / 2048; the tiny block stays finite
    assert q[20] == 6 * 352 / 2048 and np.all(np.isfinite(q)) and abs(q[3]) <= 1e-29


def test_act_quant_forward_is_a_bounded_approximation(case):
    """With act_quant the step sees quant(x) and quant(h): a real difference
    from the exact step, of the size one E2M1 digit per element allows."""
    wl, x, ids, w, W, S = case
    y, _ = oracle.moe_forward(x, ids, w, W)
    ya, _ = oracle.moe_forward(x, ids, w, W, act_quant=True)
    rel = np.abs(ya - y).max() / np.abs(y).max()
    assert 1e-6 < rel < 0.2                                      # a real, bounded approximation
