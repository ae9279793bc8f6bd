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
    wl = WORKLOADS["upper_decode"]
    ids = make_topk_ids(wl).numpy().reshape(-1)
    vals, cnt = np.unique(ids, return_counts=True)
    hist = {r: int((cnt == r).sum()) for r in set(cnt.tolist())}
    assert hist[8] == 12 and hist[4] == 12 and hist[2] >= 12 and hist[1] >= 12 - 12
    assert cnt.sum() == wl.T * wl.k


def test_zipf_routing_is_skewed():
    wl = WORKLOADS["spec_verify"]
    ids = make_topk_ids(wl).numpy().reshape(-1)
    _, cnt = np.unique(ids, return_counts=True)
    assert cnt.max() >= 8 and len(cnt) < wl.T * wl.k


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
