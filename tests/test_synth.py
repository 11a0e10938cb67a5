"""Seeded generators: determinism, row-subset draws equal to full draws, value recipes."""
import torch

from long_context_sparse_tcgen05_gb300 import synth


def test_row_subsets_equal_full_draws():
    wl = synth.WORKLOADS["prefill_128k"].replace(T=9000, S=9000, H=4, DQK=64, DV=32)
    rows = [0, 5, 4095, 4096, 8999]
    full = synth.indexer_inputs(wl, 1)
    sub = synth.indexer_rows(wl, 1, rows)
    assert torch.equal(sub["q_rows"].view(torch.uint8), full["q"][0, rows].view(torch.uint8))
    assert torch.equal(sub["q_scale_rows"], full["q_scale"][0, rows])
    assert torch.equal(sub["w_rows"], full["w"][0, rows])
    assert torch.equal(sub["k"].view(torch.uint8), full["k"].view(torch.uint8))
    at = synth.attn_inputs(wl, 2)
    ar = synth.attn_rows(wl, 2, rows)
    assert torch.equal(ar["q_rows"], at["q"][0, rows]) and torch.equal(ar["k"], at["k"])


def test_recipes():
    wl = synth.WORKLOADS["tiny_l1k"]
    ix = synth.indexer_inputs(wl, 0)
    q = ix["q"].float()
    assert q.min() >= -3 and q.max() <= 3 and torch.equal(q, q.round())
    assert ix["w"].min() >= 1 and ix["w"].max() <= 4
    ix2 = synth.indexer_inputs(wl, 0)
    assert torch.equal(ix["q"], ix2["q"])
    w8 = synth.WORKLOADS["prefill_128k"].replace(T=512, S=512)
    f = synth.indexer_inputs(w8, 0)
    assert f["q"].dtype == torch.float8_e4m3fn
    amax = (f["q"].float().abs().amax(dim=(2, 3)))
    assert torch.all(amax <= 448) and torch.all(amax >= 416)  # scale = amax / 448
    assert torch.all(f["w"] >= 0) and torch.all(f["w"] <= 1 / 8)


def test_clustered_layers_share_noise_inside_a_cluster():
    # every layer is base + 0.3 * unit noise; inside a cluster 3/4 of the noise variance is
    # shared: corr = (1 + 0.09 * 0.75) / 1.09 inside, 1 / 1.09 across clusters
    wl = synth.WORKLOADS["heatmap_128k"].replace(T=256, S=256)
    assert len(wl.clusters) == wl.n_layers == 16
    deq = []
    for l in (0, 1, 2, 6):
        ix = synth.indexer_inputs(wl, l)
        deq.append((ix["q"].float() * ix["q_scale"][..., None, None]).flatten().double())
    corr = lambda a, b: float(torch.corrcoef(torch.stack([a, b]))[0, 1])
    inside = corr(deq[1], deq[2])            # layers 1, 2: cluster 1
    across = corr(deq[0], deq[1])            # clusters 0 and 1
    assert abs(inside - (1 + 0.09 * 0.75) / 1.09) < 0.01
    assert abs(across - 1 / 1.09) < 0.01
    assert abs(corr(deq[2], deq[3]) - 1 / 1.09) < 0.01  # clusters 1 and 3
    assert abs(float(deq[3].std()) - 1.09 ** 0.5) < 0.02


def test_shared_cache_steps_share_keys_and_kv_but_not_queries():
    wl = synth.WORKLOADS["mtp_draft_b32_200k"].replace(B=2, S=300, q_pos0=300)
    g = synth.group_inputs(wl, 4, with_indexer=True)
    for l in range(1, 4):
        assert g[l]["at"]["k"] is g[0]["at"]["k"] and g[l]["ix"]["k"] is g[0]["ix"]["k"]
        assert not torch.equal(g[l]["at"]["q"], g[0]["at"]["q"])
        assert not torch.equal(g[l]["ix"]["q"].view(torch.uint8), g[0]["ix"]["q"].view(torch.uint8))
        # the same values layer_inputs draws for that step
        one = synth.layer_inputs(wl, l, with_indexer=True)
        assert torch.equal(one["at"]["k"], g[l]["at"]["k"]) and torch.equal(one["at"]["q"], g[l]["at"]["q"])
        assert torch.equal(one["ix"]["q"].view(torch.uint8), g[l]["ix"]["q"].view(torch.uint8))
        assert torch.equal(one["ix"]["k"].view(torch.uint8), g[l]["ix"]["k"].view(torch.uint8))
        assert torch.equal(one["ix"]["q_scale"], g[l]["ix"]["q_scale"])
