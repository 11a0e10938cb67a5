"""GPU checks of the boundary itself: strided operand views give the results of their dense
copies (bit for bit: the same kernels read the same values), and the workspace-size queries
hand the calls exactly the room their split schedules need (the split path is taken -- it
launches its merge kernel -- and its results are exact against the oracle)."""
import numpy as np
import pytest
import torch

import long_context_sparse_tcgen05_gb300 as dsa
import oracle
from long_context_sparse_tcgen05_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_tcgen05_gb300 import build
    build.build()
    dsa.load_library()
    dsa.read_device_flags()


def _dense(ix):
    return {k: (v.contiguous() if torch.is_tensor(v) else v) for k, v in ix.items()}


@pytest.mark.parametrize("HI,DI,dtype", [(64, 128, "bf16"), (64, 128, "e4m3"), (4, 64, "bf16")])
def test_indexer_strided_views_equal_dense(HI, DI, dtype):
    # B = 2 sequences of a 700-token cache; the call sees rows 300..539 of each sequence's
    # queries and the first 640 keys of each cache: q and k are strided views of the larger
    # tensors (token stride, sequence stride), w and the scales dense copies of the rows
    base = synth.WORKLOADS["prefill_16k"] if HI == 64 else synth.WORKLOADS["tiny_l1k"]
    wl = base.replace(B=2, T=700, S=700, idx_dtype=dtype, values="int", k=64)
    full = synth.indexer_inputs(wl, 0, DEV)
    r0, r1, S = 300, 540, 640
    view = dict(q=full["q"][:, r0:r1], k=full["k"][:, :S], w=full["w"][:, r0:r1].contiguous(),
                q_scale=None if full["q_scale"] is None else full["q_scale"][:, r0:r1].contiguous(),
                k_scale=None if full["k_scale"] is None else full["k_scale"][:, :S].contiguous(),
                q_pos0=S - (r1 - r0), diag=0)
    assert not view["q"].is_contiguous() and not view["k"].is_contiguous()
    got = dsa.dsa_topk(wl.k, ix=view)
    want = dsa.dsa_topk(wl.k, ix=_dense(view))
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    sc_v = dsa.indexer_scores(view)
    sc_d = dsa.indexer_scores(_dense(view))
    assert torch.equal(sc_v, sc_d)
    # and the oracle agrees on the integer inputs, bit for bit
    rows = [0, 1, 100, 239, 240, 300, 479]
    ref = oracle.indexer_topk(_dense(view), wl.k, rows)
    assert np.array_equal(got.reshape(-1, wl.k)[rows].cpu().numpy(), ref)
    assert dsa.read_device_flags() == 0


def _rand_idx(B, T, k, S, seed=3):
    g = torch.Generator(device=DEV).manual_seed(seed)
    idx = torch.randint(0, S, (B, T, k), generator=g, device=DEV, dtype=torch.int32)
    idx = torch.sort(idx, dim=-1).values
    idx[:, :, k - 5:] = -1  # some padding
    return idx.contiguous()


@pytest.mark.parametrize("latent", [True, False])
def test_attention_strided_views_equal_dense(latent):
    if latent:
        wl = synth.WORKLOADS["prefill_16k"].replace(B=2, T=96, S=1000, k=256)
    else:
        wl = synth.WORKLOADS["tiny_l1k"].replace(B=2, T=96, S=1000, k=64)
    at = synth.attn_inputs(wl, 0, DEV)
    r0, r1, S = 20, 84, 900
    view = dict(q=at["q"][:, r0:r1], k=at["k"][:, :S], v=None if at["v"] is None else at["v"][:, :S],
                d_v=at["d_v"], scale=at["scale"])
    dense = dict(view, q=view["q"].contiguous(), k=view["k"].contiguous(),
                 v=None if view["v"] is None else view["v"].contiguous())
    assert not view["q"].is_contiguous() and not view["k"].is_contiguous()
    idx = _rand_idx(2, r1 - r0, wl.k, S)
    o1, l1 = dsa.dsa_sparse_attn(view, idx)
    o2, l2 = dsa.dsa_sparse_attn(dense, idx)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rows = [0, 5, 63, 64, 100, 127]
    host = dict(q_rows=dense["q"].reshape(-1, wl.H, wl.DQK)[rows].cpu(), k=dense["k"].cpu(),
                v=None if dense["v"] is None else dense["v"].cpu(), d_v=wl.DV, scale=wl.scale, T=r1 - r0)
    ref_o, _ = oracle.sparse_attn(host, idx.reshape(-1, wl.k)[rows].cpu().numpy(), rows)
    err = np.abs(o1.reshape(-1, wl.H, wl.DV)[rows].float().cpu().numpy() - ref_o).max()
    assert err <= 2e-2
    assert dsa.read_device_flags() == 0


def _launches(fn):
    torch.cuda.synchronize()
    n0 = dsa.launch_count()
    out = fn()
    torch.cuda.synchronize()
    return out, dsa.launch_count() - n0


def test_topk_workspace_query_selects_the_split_path():
    # 12 long rows: the few-long-rows path only with the queried room
    R, n, k = 12, 200000, 2048
    sc = synth.scores_input(R, n, DEV, "int", lo=-40, hi=40)
    q_pos0 = n - R
    need = dsa.topk_workspace_size(1, R, n, q_pos0, 0, k)
    assert need > dsa.WS_MIN
    ref = oracle.topk_rows(sc.double().cpu().numpy(), np.clip(np.arange(R) + q_pos0, 0, n), k)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    idx, nl = _launches(lambda: dsa.dsa_topk(k, scores=sc[None], q_pos0=q_pos0, ws=ws))
    # few long rows in the queried room: sampled threshold, filter, candidate top-k, and the
    # gated pass for rows the candidates could not finish
    assert nl == 4
    assert np.array_equal(idx[0].cpu().numpy(), ref)
    ws_min = torch.zeros(dsa.WS_MIN, dtype=torch.uint8, device=DEV)
    idx2, nl2 = _launches(lambda: dsa.dsa_topk(k, scores=sc[None], q_pos0=q_pos0, ws=ws_min))
    assert nl2 == 1
    assert np.array_equal(idx2[0].cpu().numpy(), ref)
    ws_short = torch.zeros(need - 4, dtype=torch.uint8, device=DEV)
    _, nl3 = _launches(lambda: dsa.dsa_topk(k, scores=sc[None], q_pos0=q_pos0, ws=ws_short))
    assert nl3 == 1


def test_attention_workspace_query_selects_the_split_path():
    wl = synth.WORKLOADS["decode_b32_200k"].replace(B=8, S=30000, q_pos0=30000)
    at = synth.attn_inputs(wl, 0, DEV)
    idx = _rand_idx(8, 1, 2048, 30000, seed=9)
    need = dsa.attn_workspace_size(at, 2048)
    assert need > dsa.WS_MIN
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    (o1, l1), nl = _launches(lambda: dsa.dsa_sparse_attn(at, idx, ws=ws))
    assert nl == 2  # parts, then the combine
    ws_min = torch.zeros(dsa.WS_MIN, dtype=torch.uint8, device=DEV)
    (o2, l2), nl2 = _launches(lambda: dsa.dsa_sparse_attn(at, idx, ws=ws_min))
    assert nl2 == 1
    rows = list(range(8))
    host = dict(q_rows=at["q"].reshape(-1, wl.H, wl.DQK).cpu(), k=at["k"].cpu(), v=None, d_v=wl.DV,
                scale=wl.scale, T=1)
    ref_o, ref_l = oracle.sparse_attn(host, idx.reshape(-1, 2048).cpu().numpy(), rows)
    for o, l in ((o1, l1), (o2, l2)):
        assert np.abs(o.reshape(-1, wl.H, wl.DV).float().cpu().numpy() - ref_o).max() <= 2e-2
        assert np.abs(l.reshape(-1, wl.H).cpu().numpy() - ref_l).max() <= 1e-3


def test_group_workspace_query_covers_decode_attention_splits():
    wl = synth.WORKLOADS["decode_b32_200k"].replace(B=4, S=100000, q_pos0=100000)
    layers = synth.group_inputs(wl, 4, DEV)
    dsa.release_workspace()
    (outs, lses, bufs), nl = _launches(lambda: dsa.indexshare_group_forward(layers, "FSSS", wl.k))
    # indexer + split top-k (segments + merge) + the four layers in one split attention launch
    # (parts + combine): the workspace the query sized holds every part of all four layers
    assert nl == 1 + 2 + 2
    rows = list(range(4))
    ref = oracle.group_forward([{k: v for k, v in l.items()} for l in layers], "FSSS", wl.k, rows)
    got = bufs[0].reshape(-1, wl.k).cpu().numpy()
    rec = np.mean([len(np.intersect1d(g[g >= 0], e[e >= 0])) / max(1, (e >= 0).sum()) for g, e in zip(got, ref[0]["idx"])])
    assert rec >= 0.999
    assert dsa.read_device_flags() == 0
