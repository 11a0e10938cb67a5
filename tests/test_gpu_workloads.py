"""Full-size workloads through the same call the benchmark times (one F,S,S,S group via
indexshare_group_forward), checked against the oracle on sampled query rows.

Index rows: bit-exact on the small-integer workload; recall >= 0.999 plus validity (every
selected position scores within the fp32 rounding bound of the oracle's k-th score) on the
Gaussian ones.  Attention: the oracle recomputes each sampled row over the GPU's own index
row (so near-ties of the selection do not leak into the attention check); max-abs <= 2e-2.
"""
import numpy as np
import pytest
import torch

import long_context_sparse_tcgen05_gb300 as dsa
import oracle
from long_context_sparse_tcgen05_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_tcgen05_gb300 import build
    build.build()
    dsa.load_library()
    dsa.read_device_flags()


def _subset_batches(d: dict, keys, bsel):
    out = dict(d)
    for k in keys:
        if out.get(k) is not None:
            out[k] = out[k][bsel].contiguous()
    return out


@pytest.mark.parametrize("name,n_rows", [("tiny_l1k", 1024), ("prefill_16k", 48), ("prefill_128k", 24),
                                         ("decode_b32_200k", 8), ("chunked_prefill_1m", 12),
                                         ("mtp_draft_b32_200k", 8)])
def test_workload_group_sampled_rows(name, n_rows):
    wl = synth.WORKLOADS[name]
    layers = synth.group_inputs(wl, 4, DEV)
    outs, lses, bufs = dsa.indexshare_group_forward(layers, "FSSS", wl.k)
    torch.cuda.synchronize()
    assert dsa.read_device_flags() == 0
    idx = bufs[0].reshape(wl.B * wl.T, wl.k)

    if wl.B > 1:  # decode: check whole sequences (one row each), a few of them
        bsel = torch.linspace(0, wl.B - 1, n_rows).long().tolist()
        rows = bsel
        ix = _subset_batches(layers[0]["ix"], ["q", "w", "q_scale", "k", "k_scale"], bsel)
        ats = [_subset_batches(l["at"], ["q", "k", "v"], bsel) for l in layers]
        orc_rows = list(range(len(bsel)))
    else:
        rows = synth.sample_rows(wl, n_rows)
        ix, ats, orc_rows = layers[0]["ix"], [l["at"] for l in layers], rows

    got_idx = idx[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    ref_idx, ref_sc = oracle.indexer_topk(ix, wl.k, orc_rows, return_scores=True)
    if wl.values == "int":
        assert np.array_equal(got_idx, ref_idx)
    else:
        nv = oracle.row_visible(ix, orc_rows)
        recalls = []
        for r in range(len(rows)):
            g = got_idx[r][got_idx[r] >= 0]
            e = ref_idx[r][ref_idx[r] >= 0]
            assert len(g) == len(e) and np.all(np.diff(g) > 0) and np.all(g < nv[r])
            recalls.append(len(np.intersect1d(g, e)) / len(e) if len(e) else 1.0)
            if 0 < len(e) < nv[r]:
                tau = np.sort(ref_sc[r, :nv[r]])[::-1][len(e) - 1]
                assert ref_sc[r, g].min() >= tau - 1e-4 * abs(tau)
        assert np.mean(recalls) >= 0.999, (np.mean(recalls), np.min(recalls))

    for l in range(4):
        ref_o, ref_l = oracle.sparse_attn(ats[l], got_idx, orc_rows)
        o = outs[l].reshape(wl.B * wl.T, wl.H, wl.DV)[torch.as_tensor(rows, device=DEV)].float().cpu().numpy()
        assert np.abs(o - ref_o).max() <= 2e-2, (l, np.abs(o - ref_o).max())
        gl = lses[l].reshape(wl.B * wl.T, wl.H)[torch.as_tensor(rows, device=DEV)].cpu().numpy()
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - ref_l[fin]).max() <= 1e-3
    del layers, outs, lses, bufs
    torch.cuda.empty_cache()


def test_draft_steps_in_one_launch_at_full_size():
    """indexshare_draft_forward at the 32 x 200,000 draft shape: the first step's indexer +
    top-k, then one attention launch in which the four draft queries of each sequence attend
    over its one index row.  Integer indexer operands make the selection exact, so sampled
    sequences are compared with the oracle's draft walk directly (index rows bit for bit,
    outputs within 2e-2, LSE within 1e-3); the selection equals dsa_topk on the first step and
    every step equals its own attention call over it (within 1e-2, the decode split of a
    single step sums in another order)."""
    wl = synth.WORKLOADS["mtp_draft_b32_200k"].replace(values="int")
    layers = synth.group_inputs(wl, 4, DEV, with_indexer=True)
    at = dict(layers[0]["at"])
    at["q"] = torch.cat([l["at"]["q"] for l in layers], dim=1).contiguous()
    out, lse, idx = dsa.indexshare_draft_forward(layers[0]["ix"], at, wl.k)
    torch.cuda.synchronize()
    assert dsa.read_device_flags() == 0
    idx_f = dsa.dsa_topk(wl.k, ix=layers[0]["ix"])
    assert torch.equal(idx_f.reshape(wl.B, wl.k), idx.reshape(wl.B, wl.k))
    for s in range(4):
        o_s, l_s = dsa.dsa_sparse_attn(layers[s]["at"], idx_f)
        assert (o_s[:, 0].float() - out[:, s].float()).abs().max().item() <= 1e-2
        assert (l_s[:, 0] - lse[:, s]).abs().max().item() <= 1e-3
    bsel = [0, 13, 31]
    ix = _subset_batches(layers[0]["ix"], ["q", "w", "q_scale", "k", "k_scale"], bsel)
    ats = _subset_batches(at, ["q", "k", "v"], bsel)
    ref_idx, ref_o, ref_l = oracle.draft_forward(ix, ats, wl.k)
    assert np.array_equal(idx.reshape(wl.B, wl.k)[bsel].cpu().numpy(), ref_idx)
    assert np.abs(out[bsel].float().cpu().numpy() - ref_o).max() <= 2e-2
    gl, fin = lse[bsel].cpu().numpy(), np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(gl), fin) and np.abs(gl[fin] - ref_l[fin]).max() <= 1e-3
    del layers, at, out, lse, idx, idx_f
    torch.cuda.empty_cache()


def test_heatmap_all_full_pass_and_overlap_matrix_sampled_rows():
    """The launch configuration of bench.py --heatmap: 16 layers of the 128K clustered
    workload, each with its own indexer + top-k, then the all-pairs overlap matrix.  Per layer
    the index rows of three sampled queries are checked against the oracle (recall, validity);
    the matrix's per-row intersection counts are checked exactly on sampled rows against set
    intersections of the GPU's own index rows, and its means against the mean over all rows
    of count / valid count computed from those counts."""
    wl = synth.WORKLOADS["heatmap_128k"]
    n, R, k = wl.n_layers, wl.B * wl.T, wl.k
    check_rows = [5, 2048, 20000]
    bufs = []
    for l in range(n):
        ix = synth.indexer_inputs(wl, l, DEV)
        bufs.append(dsa.dsa_topk(k, ix=ix))
        got = bufs[-1].reshape(R, k)[torch.as_tensor(check_rows, device=DEV)].cpu().numpy()
        ref, _ = oracle.indexer_topk(ix, k, check_rows, return_scores=True)
        rec = [len(np.intersect1d(g[g >= 0], e[e >= 0])) / max(1, (e >= 0).sum()) for g, e in zip(got, ref)]
        assert np.mean(rec) >= 0.999, (l, rec)
        del ix
        torch.cuda.empty_cache()
    M, cnt = dsa.topk_overlap_matrix(bufs, counts=True)
    assert dsa.read_device_flags() == 0
    rows = synth.sample_rows(wl, 12)
    sel = torch.as_tensor(rows, device=DEV)
    host = [b.reshape(R, k)[sel].cpu().numpy() for b in bufs]
    c = cnt[sel].cpu().numpy()
    for r in range(len(rows)):
        sets = [set(h[r][h[r] >= 0].tolist()) for h in host]
        want = np.array([[len(sets[i] & sets[j]) for j in range(n)] for i in range(n)])
        assert np.array_equal(c[r], want), rows[r]
    # means: the matrix equals the mean of count/valid over all rows
    cf = cnt.double()
    diag = torch.diagonal(cf, dim1=1, dim2=2)[:, :, None]
    frac = torch.where(diag == 0, torch.ones_like(cf), cf / diag.clamp(min=1))
    np.testing.assert_allclose(np.array(M), frac.mean(0).cpu().numpy(), rtol=1e-9, atol=0)
    # clusters: (1,2), (3,4,5), (6..15) overlap more inside than across
    assert M[1][2] > M[0][1] and M[4][5] > M[2][3] and M[7][8] > M[5][6]
    del bufs, cnt
    torch.cuda.empty_cache()


def test_fp8_append_of_the_128k_queries_sampled_rows():
    """The launch configuration of bench.py --kernel quant: the queries of 131,072 tokens
    (64 heads x 128 dims, one scale per token) quantised into a cache in one call; sampled
    tokens bit-exact against the oracle's quantiser."""
    T, width = 131072, 64 * 128
    g = torch.Generator(device=DEV)
    g.manual_seed(synth.SEED_BASE + 17)
    x = torch.randn((1, T, width), generator=g, device=DEV).to(torch.bfloat16)
    codes = torch.empty((1, T, width), dtype=torch.uint8, device=DEV)
    scales = torch.empty((1, T), dtype=torch.float32, device=DEV)
    dsa.dsa_quantize_e4m3_append(x, codes, scales)
    assert dsa.read_device_flags() == 0
    rows = torch.as_tensor([0, 1, 4095, 65536, 99999, T - 1], device=DEV)
    want_c, want_s = oracle.quantize_e4m3_rows(x[0, rows], width)
    assert np.array_equal(codes[0, rows].cpu().numpy(), want_c)
    assert np.array_equal(scales[0, rows].cpu().numpy(), want_s)


def test_packed_prompts_equal_each_prompt_alone():
    """Three prompts of 16K, 4K and 1K tokens of the 128K workload's operands in one packed
    call: every output, LSE and index row equals the prompt's own call bit for bit."""
    base = synth.WORKLOADS["prefill_128k"]
    lens = [16384, 4096, 1024]
    per = [synth.group_inputs(base.replace(T=n, S=n, q_pos0=0, wid=40 + i), 4, DEV) for i, n in enumerate(lens)]
    packed = []
    for l in range(4):
        at = dict(per[0][l]["at"])
        at["q"] = torch.cat([p[l]["at"]["q"] for p in per], dim=1)
        at["k"] = torch.cat([p[l]["at"]["k"] for p in per], dim=1)
        ix = None
        if l == 0:
            ix = dict(per[0][0]["ix"])
            for key in ("q", "w", "q_scale", "k", "k_scale"):
                ix[key] = torch.cat([p[0]["ix"][key] for p in per], dim=1)
        packed.append(dict(ix=ix, at=at))
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    outs, lses, bufs = dsa.indexshare_group_forward_varlen(packed, "FSSS", base.k, cu, cu, [0, 0, 0])
    torch.cuda.synchronize()
    assert dsa.read_device_flags() == 0
    for i, p in enumerate(per):
        o1, l1, b1 = dsa.indexshare_group_forward(p, "FSSS", base.k)
        r0, r1 = cu[i], cu[i + 1]
        assert torch.equal(bufs[0][:, r0:r1], b1[0])
        for l in range(4):
            assert torch.equal(outs[l][:, r0:r1], o1[l]) and torch.equal(lses[l][:, r0:r1], l1[l])
    del per, packed, outs, lses, bufs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,dtype,n_rows", [("prefill_128k", "e4m3", 24), ("prefill_128k", "bf16", 12),
                                               ("decode_b32_200k", "e4m3", 32), ("chunked_prefill_1m", "e4m3", 10)])
def test_indexer_topk_bit_exact_at_full_size_on_integer_operands(name, dtype, n_rows):
    """The indexer -> top-k path at each workload's full shape, in the launch configuration the
    group call uses (row chunks of the score workspace at 128K, the key-range split of the
    decode indexer with the split top-k over 200,000-key rows, 1M-key rows), on small-integer
    operands: q_I, k_I in [-3, 3], w in [1, 4], so every score is an integer of magnitude at most
    64 * 4 * 128 * 9 = 294,912 < 2^24 and exact in fp32.  Sampled index rows must equal the
    oracle's bit for bit, ties to the lower position included."""
    wl = synth.WORKLOADS[name].replace(values="int", idx_dtype=dtype)
    ix = synth.indexer_inputs(wl, 0, DEV)
    idx = dsa.dsa_topk(wl.k, ix=ix)
    torch.cuda.synchronize()
    assert dsa.read_device_flags() == 0
    rows = synth.sample_rows(wl, n_rows) if wl.B == 1 else list(range(wl.B))
    # rows on both sides of seams: the selecting path's row chunks (14,592 rows at 128K on a
    # 152-SM part) and the score buffer's 8,192-row chunks
    if name == "prefill_128k":
        rows = sorted(set(rows) | {8191, 8192, 14591, 14592, 65535, 65536, 116735, 116736})
    got = idx.reshape(wl.B * wl.T, wl.k)[torch.as_tensor(rows, device=DEV)].cpu().numpy()
    ref = oracle.indexer_topk(ix, wl.k, rows)
    assert np.array_equal(got, ref)
    del ix, idx
    torch.cuda.empty_cache()
