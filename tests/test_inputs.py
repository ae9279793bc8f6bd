"""Host-side checks of the seeded input recipe (no GPU)."""
import numpy as np
import torch

import oracle
from quantized_moe_routed_gb300.inputs import (WORKLOADS, Workload, algorithmic_bytes, make_topk_ids,
                                               make_topk_w, make_x, quantize_nvfp4, rotate_ids,
                                               rotation_delta, touched_experts)


def test_workload_shapes_and_determinism():
    for name, wl in WORKLOADS.items():
        ids = make_topk_ids(wl)
        assert ids.shape == (wl.T, wl.k) and ids.dtype == torch.int32
        assert torch.equal(ids, make_topk_ids(wl))
        for t in range(wl.T):                       # distinct within a token
            assert len(set(ids[t].tolist())) == wl.k
        assert int(ids.min()) >= 0 and int(ids.max()) < wl.E
        w = make_topk_w(wl)
        assert torch.allclose(w.double().sum(1), torch.ones(wl.T, dtype=torch.float64), atol=1e-6)
        assert bool((w > 0).all())
    x = make_x(WORKLOADS["decode"])
    assert x.dtype == torch.bfloat16 and x.shape == (1, 4096)
    assert abs(float(x.float().std()) - 1.0) < 0.05


def test_class_routing_hits_exact_classes():
    """12 experts in each class R_e = 8, 4, 2, 1 (180 picks), then 12 filler
    picks over the other experts: here each filler lands on its own expert."""
    wl = WORKLOADS["upper_decode"]
    ids = make_topk_ids(wl).numpy().reshape(-1)
    vals, cnt = np.unique(ids, return_counts=True)
    hist = {r: int((cnt == r).sum()) for r in set(cnt.tolist())}
    assert hist == {8: 12, 4: 12, 2: 12, 1: 24}
    assert int(cnt[(cnt != 8) & (cnt != 4)].sum()) == 12 * 2 + 12 * 1 + 12
    assert cnt.sum() == wl.T * wl.k and len(vals) == 60


def test_zipf_routing_is_skewed():
    """Zipf(1) ranks, drawn without replacement per token: the hottest expert
    takes 13 of the 16 tokens (R_e up to 13, not 1-8), 62 experts touched."""
    wl = WORKLOADS["spec_verify"]
    ids = make_topk_ids(wl).numpy().reshape(-1)
    _, cnt = np.unique(ids, return_counts=True)
    assert int(cnt.max()) == 13 and len(cnt) == 62
    assert int((cnt == 1).sum()) == 39     # a long tail of single-pair experts


def test_quantizer_random_error_bound():
    """Every dequantised weight lies within half an E2M1 step (times its block
    scale) of the fp32 source, and codes respect the format."""
    g = torch.Generator().manual_seed(0)
    w = torch.randn((64, 256), generator=g) * 0.02
    q, s, ts = quantize_nvfp4(w)
    back = oracle.dequant(q, s, float(ts))
    scale = s.view(torch.float8_e4m3fn).to(torch.float64).repeat_interleave(16, 1).numpy() * float(ts)
    err = np.abs(back - w.double().numpy())
    # largest E2M1 gap is 2 (between 4 and 6): half-gap 1 in block-scale units
    assert np.all(err <= 1.0 * scale + 1e-30)
    assert float(ts) > 0 and int(s.max()) <= 0x7E


def test_quantizer_zero_matrix():
    q, s, ts = quantize_nvfp4(torch.zeros((4, 32)))
    assert float(ts) == 1.0 and int(q.max()) == 0 and int(s.max()) == 0


def test_rotation_keeps_histogram_and_disjointness():
    wl = WORKLOADS["decode"]
    ids = make_topk_ids(wl)
    d = rotation_delta(ids, wl.E)
    sets = [set(rotate_ids(ids, s, d, wl.E).reshape(-1).tolist()) for s in range(4)]
    for a in range(4):
        for b in range(a + 1, 4):
            assert sets[a].isdisjoint(sets[b])
    r = rotate_ids(ids, 3, d, wl.E)
    assert sorted(np.unique(r.numpy(), return_counts=True)[1]) == sorted(np.unique(ids.numpy(), return_counts=True)[1])


def test_algorithmic_bytes_decode():
    wl = WORKLOADS["decode"]
    ids = make_topk_ids(wl)
    per_expert = 3 * 1024 * 4096 // 2 + 3 * 1024 * 4096 // 16 + 12
    assert per_expert == 7_077_900
    assert algorithmic_bytes(wl, ids) == 8 * per_expert + 4096 * 2 + 8 * 8 + 4096 * 4
    assert touched_experts(torch.tensor([[3, -1, 9, 3]]), 8) == [3]


def test_zipf_draws_follow_one_over_rank_without_replacement():
    """Reading c12 (sequential draws without replacement, p(rank r) ~ 1/r,
    rank -> expert through a seeded permutation): over many tokens the first
    pick's rank frequency is p_r, and the (first, second) pair frequency is
    p_r1 * p_r2 / (1 - p_r1), each within 5 binomial standard deviations."""
    from quantized_moe_routed_gb300.inputs import _ids_zipf, _np_rng
    E, n = 4, 40000
    ids = _ids_zipf(_np_rng(5, 3), n, 2, E)
    perm = _np_rng(5, 3).permutation(E)        # the first thing the draw takes from its stream
    rank_of = np.empty(E, np.int64)
    rank_of[perm] = np.arange(E)
    r1, r2 = rank_of[ids[:, 0]], rank_of[ids[:, 1]]
    assert np.all(r1 != r2)
    p = 1.0 / np.arange(1, E + 1)
    p /= p.sum()
    f1 = np.bincount(r1, minlength=E) / n
    assert np.all(np.abs(f1 - p) < 5 * np.sqrt(p * (1 - p) / n))
    joint = np.zeros((E, E))
    np.add.at(joint, (r1, r2), 1.0 / n)
    for a in range(E):
        for b in range(E):
            q = 0.0 if a == b else p[a] * p[b] / (1 - p[a])
            assert abs(joint[a, b] - q) <= 5 * np.sqrt(q * (1 - q) / n) + 1e-12, (a, b, joint[a, b], q)


def test_router_logits_are_seeded_and_leave_the_other_streams_alone():
    from quantized_moe_routed_gb300.inputs import make_router_logits
    wl = WORKLOADS["spec_verify"]
    a = make_router_logits(wl)
    assert a.shape == (wl.T, wl.E) and a.dtype == torch.float32
    assert torch.equal(a, make_router_logits(wl))
    assert not torch.equal(a, make_router_logits(wl.replace(seed=1)))
    assert abs(float(a.std()) - 1.0) < 0.05
    # x, the routing weights and the ids come from their own streams, as before
    x0, w0, i0 = make_x(wl), make_topk_w(wl), make_topk_ids(wl)
    make_router_logits(wl)
    assert torch.equal(x0, make_x(wl)) and torch.equal(w0, make_topk_w(wl)) and torch.equal(i0, make_topk_ids(wl))
