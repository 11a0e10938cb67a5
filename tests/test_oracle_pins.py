"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a closed form, a library routine, a hand-worked
example under tests/golden/, a brute-force enumeration or an invariant, chosen so that a
dropped term, a wrong sign or index, or a transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_tcgen05_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF = float("-inf")


def _ix(q, k, w, diag=0, q_pos0=0, q_scale=None, k_scale=None):
    return dict(q=q, k=k, w=w, diag=diag, q_pos0=q_pos0, q_scale=q_scale, k_scale=k_scale)


# --- number formats ------------------------------------------------------------------

def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ours = oracle.e4m3_to_double(codes)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_bf16_decode_all_codes_match_torch():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ours = oracle.bf16_to_double(codes)
    ref = codes.view(torch.bfloat16).float().double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# --- indexer scores ------------------------------------------------------------------

def test_indexer_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "indexer_tiny.json")))
    q = torch.tensor(g["q"], dtype=torch.float32)[None].to(torch.bfloat16)
    k = torch.tensor(g["k"], dtype=torch.float32)[None].to(torch.bfloat16)
    w = torch.tensor(g["w"], dtype=torch.float32)[None]
    for diag in (0, 1):
        sc = oracle.indexer_scores(_ix(q, k, w, diag=diag))
        want = np.array([[NEG_INF if v is None else v for v in row] for row in g[f"scores_diag{diag}"]])
        assert np.array_equal(sc, want), (diag, sc)
        for kk in (1, 2):
            idx = oracle.indexer_topk(_ix(q, k, w, diag=diag), kk)
            assert idx.tolist() == g[f"topk_k{kk}_diag{diag}"], (diag, kk, idx)


def _rand_bf16(shape, seed, lo=None, hi=None):
    g = torch.Generator().manual_seed(seed)
    if lo is not None:
        return torch.randint(lo, hi + 1, shape, generator=g).float().to(torch.bfloat16)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def test_indexer_single_head_unit_weight_is_relu_matmul():
    """H_I = 1, w = 1: I = ReLU(q k^T) on the visible triangle (library matmul)."""
    T, DI = 37, 16
    q = _rand_bf16((1, T, 1, DI), 1)
    k = _rand_bf16((1, T, DI), 2)
    w = torch.ones(1, T, 1)
    sc = oracle.indexer_scores(_ix(q, k, w))
    ref = torch.relu(q[0, :, 0].double() @ k[0].double().T).numpy()
    mask = np.tril(np.ones((T, T), dtype=bool), -1)  # s < t
    assert np.all(np.isneginf(sc[~mask]))
    np.testing.assert_allclose(sc[mask], ref[mask], rtol=1e-12, atol=1e-12)


def test_indexer_head_terms_and_linearity_in_w():
    """A one-hot w picks ReLU(q_h k^T) of that head alone (library matmul, checks the head
    index and operand orientation); the score is linear in w (so no head term is dropped
    or double counted)."""
    T, HI, DI = 29, 5, 8
    q = _rand_bf16((1, T, HI, DI), 3)
    k = _rand_bf16((1, T, DI), 4)
    mask = np.tril(np.ones((T, T), dtype=bool), -1)
    for h in range(HI):
        w = torch.zeros(1, T, HI)
        w[..., h] = 1.0
        sc = oracle.indexer_scores(_ix(q, k, w))
        ref = torch.relu(q[0, :, h].double() @ k[0].double().T).numpy()
        np.testing.assert_allclose(sc[mask], ref[mask], rtol=1e-12, atol=1e-12)
    g = torch.Generator().manual_seed(5)
    w1 = torch.rand(1, T, HI, generator=g)
    w2 = torch.randn(1, T, HI, generator=g)  # negative weights allowed
    a, b = 0.75, -2.5
    s1 = oracle.indexer_scores(_ix(q, k, w1))
    s2 = oracle.indexer_scores(_ix(q, k, w2))
    s12 = oracle.indexer_scores(_ix(q, k, (a * w1.double() + b * w2.double()).float()))
    w12 = (a * w1.double() + b * w2.double()).float().double()
    # recompute a*s1 + b*s2 with the fp32-rounded combined weight via per-head terms
    terms = [oracle.indexer_scores(_ix(q, k, torch.nn.functional.one_hot(torch.full((1, T), h), HI).float()))
             for h in range(HI)]
    with np.errstate(invalid="ignore"):  # -inf * 0 on the masked triangle
        comb = sum(w12[0, :, h].numpy()[:, None] * terms[h] for h in range(HI))
        lin = a * s1 + b * s2
    np.testing.assert_allclose(s12[mask], comb[mask], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(s12[mask], lin[mask], rtol=1e-5, atol=1e-4)


def test_indexer_integer_inputs_exact_closed_form():
    """Small-integer operands: the score is an integer, below 2^24, reproduced exactly by
    exact integer arithmetic over every (t, h, s)."""
    wl = synth.WORKLOADS["tiny_l1k"].replace(T=96, S=96)
    ix = synth.indexer_inputs(wl, 0)
    sc = oracle.indexer_scores(ix)
    qi = ix["q"].float().numpy().astype(np.int64)[0]   # [T,HI,DI]
    ki = ix["k"].float().numpy().astype(np.int64)[0]   # [S,DI]
    wi = ix["w"].numpy().astype(np.int64)[0]           # [T,HI]
    dots = np.einsum("thd,sd->ths", qi, ki)
    ref = np.einsum("th,ths->ts", wi, np.maximum(dots, 0))
    mask = np.tril(np.ones((96, 96), dtype=bool), -1)
    assert np.array_equal(sc[mask], ref[mask].astype(np.float64))
    assert np.abs(ref).max() < 2 ** 24


def test_indexer_fp8_scales_fold_out():
    """ReLU(c x) = c ReLU(x) for c > 0: per-token scales multiply the unit-scale score."""
    wl = synth.WORKLOADS["prefill_128k"].replace(T=64, S=64, values="gauss")
    ix = synth.indexer_inputs(wl, 0)
    sc = oracle.indexer_scores(ix)
    unit = dict(ix, q_scale=torch.ones_like(ix["q_scale"]), k_scale=torch.ones_like(ix["k_scale"]))
    su = oracle.indexer_scores(unit)
    f = ix["q_scale"][0].double().numpy()[:, None] * ix["k_scale"][0].double().numpy()[None, :]
    mask = np.tril(np.ones((64, 64), dtype=bool), -1)
    np.testing.assert_allclose(sc[mask], (su * f)[mask], rtol=1e-12)
    # the e4m3 operand values are torch's own decode of the codes
    qd = ix["q"].float().double()[0, 5, 2] * ix["q_scale"][0, 5].double()
    kd = ix["k"].float().double()[0, 3] * ix["k_scale"][0, 3].double()
    one = torch.zeros(1, 64, 64)
    one[0, 5, 2] = 1.0
    s1 = oracle.indexer_scores(dict(ix, w=one), rows=[5])
    assert s1[0, 3] == pytest.approx(max(0.0, float(qd @ kd)), rel=1e-12)


def test_indexer_visibility_rule():
    T = 20
    q = _rand_bf16((2, T, 2, 8), 6, -2, 2)
    k = _rand_bf16((2, T + 5, 8), 7, -2, 2)
    w = torch.ones(2, T, 2)
    for diag, q_pos0 in ((0, 0), (1, 0), (0, 5), (1, 3)):
        sc = oracle.indexer_scores(_ix(q, k, w, diag=diag, q_pos0=q_pos0))
        for r in range(2 * T):
            n = min(T + 5, max(0, r % T + q_pos0 + diag))
            assert not np.isneginf(sc[r, :n]).any()
            assert np.isneginf(sc[r, n:]).all()
    assert oracle.visible(10, 3, 0) == 3 and oracle.visible(10, 3, 1) == 4
    assert oracle.visible(10, 30, 1) == 10 and oracle.visible(10, 0, 0) == 0


# --- top-k ---------------------------------------------------------------------------

def _brute_topk(row, n, k):
    order = sorted(range(n), key=lambda s: (-row[s], s))
    sel = sorted(order[:k])
    return sel + [-1] * (k - len(sel))


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_full_sort_with_heavy_ties(seed):
    g = torch.Generator().manual_seed(100 + seed)
    R, L = 40, 64
    sc = torch.randint(-1, 2, (R, L), generator=g).double().numpy()
    if seed % 2:
        sc = sc + 0.5 * torch.randint(0, 2, (R, L), generator=g).double().numpy()
    n_valid = torch.randint(0, L + 1, (R,), generator=g).numpy()
    for k in (1, 3, 16, 63, 64, 80):
        idx = oracle.topk_rows(sc, n_valid, k)
        for r in range(R):
            assert idx[r].tolist() == _brute_topk(sc[r].tolist(), int(n_valid[r]), k)


def test_topk_invariants_on_gaussian_rows():
    g = torch.Generator().manual_seed(9)
    R, L, k = 16, 3000, 257
    sc = torch.randn(R, L, generator=g).double().numpy()
    n_valid = np.array([0, 1, 200, 256, 257, 258] + [L] * (R - 6))
    idx = oracle.topk_rows(sc, n_valid, k)
    for r in range(R):
        n = int(n_valid[r])
        m = min(n, k)
        row = idx[r]
        assert (row[m:] == -1).all() and (row[:m] >= 0).all() and (row[:m] < n).all()
        assert (np.diff(row[:m]) > 0).all()
        if n > k:
            sel = np.zeros(n, bool)
            sel[row[:m]] = True
            assert sc[r, :n][sel].min() >= sc[r, :n][~sel].max()


def test_topk_zero_sign_and_nan_ranking():
    row = np.array([-0.0, 0.0, np.nan, -1.0, np.nan, 0.0])
    assert oracle.topk_rows(row, 6, 3).tolist() == [[0, 1, 5]]       # -0 ties +0
    assert oracle.topk_rows(row, 6, 5).tolist() == [[0, 1, 2, 3, 5]]  # NaN below -1
    assert oracle.topk_rows(row, 6, 6).tolist() == [[0, 1, 2, 3, 4, 5]]


# --- sparse attention ----------------------------------------------------------------

def test_attention_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "attention_tiny.json")))
    at = dict(q=torch.tensor(g["q"]).reshape(1, 1, 1, 1).to(torch.bfloat16),
              k=torch.tensor(g["k"]).reshape(1, 2, 1).to(torch.bfloat16),
              v=torch.tensor(g["v"]).reshape(1, 2, 1).to(torch.bfloat16), d_v=1, scale=g["scale"])
    out, lse = oracle.sparse_attn(at, np.array([g["idx"]], dtype=np.int32))
    assert out[0, 0, 0] == pytest.approx(g["out"], abs=1e-12)
    assert lse[0, 0] == pytest.approx(g["lse"], abs=1e-12)


@pytest.mark.parametrize("latent", [False, True])
def test_attention_equals_dense_causal_when_k_covers_all(latent):
    """With n_t <= k every visible key is selected, so sparse attention is dense
    strictly-causal attention (library SDPA in float64)."""
    T, H, DQK, DV = 24, 3, 16, 8
    q = _rand_bf16((1, T, H, DQK), 10)
    kv = _rand_bf16((1, T, DQK), 11)
    v = None if latent else _rand_bf16((1, T, DV), 12)
    at = dict(q=q, k=kv, v=v, d_v=DV, scale=0.3)
    kk = 32
    idx = np.full((T, kk), -1, np.int32)
    for t in range(T):
        idx[t, :t] = np.arange(t)
    out, lse = oracle.sparse_attn(at, idx)
    Q = q[0].double().permute(1, 0, 2)             # [H,T,DQK]
    K = kv[0].double()[None].expand(H, T, DQK)
    V = (kv[0, :, :DV] if latent else v[0]).double()[None].expand(H, T, DV)
    mask = torch.tril(torch.ones(T, T, dtype=torch.bool), -1)
    ref = torch.nn.functional.scaled_dot_product_attention(Q[:, 1:], K, V, attn_mask=mask[1:],
                                                           scale=0.3)
    np.testing.assert_allclose(out[1:], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    z = 0.3 * (Q @ K.transpose(1, 2))
    ref_lse = torch.logsumexp(z.masked_fill(~mask, float("-inf")), dim=-1)  # [H,T]
    np.testing.assert_allclose(lse[1:], ref_lse.T[1:].numpy(), rtol=1e-12)
    # row 0 sees nothing
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()


def test_attention_single_key_and_constant_values():
    T, H, D = 6, 2, 8
    q = _rand_bf16((1, T, H, D), 13)
    kv = _rand_bf16((1, 10, D), 14)
    at = dict(q=q, k=kv, v=None, d_v=D, scale=1.0)
    idx = np.array([[j, -1, -1] for j in range(T)], np.int32)
    out, lse = oracle.sparse_attn(at, idx)
    for t in range(T):
        np.testing.assert_array_equal(out[t, 0], kv[0, t].double().numpy())
        z = float(q[0, t, 1].double() @ kv[0, t].double())
        assert lse[t, 1] == pytest.approx(z, abs=1e-12)
    const = torch.full((1, 10, D), 1.5).to(torch.bfloat16)
    idx2 = np.array([[0, 3, 9, -1, 4]] * T, np.int32)
    out2, _ = oracle.sparse_attn(dict(at, k=_rand_bf16((1, 10, D), 15), v=const), idx2)
    np.testing.assert_allclose(out2, 1.5, rtol=1e-12)


def test_attention_rejects_out_of_range_index():
    at = dict(q=_rand_bf16((1, 1, 1, 4), 16), k=_rand_bf16((1, 4, 4), 17), v=None, d_v=4, scale=1.0)
    with pytest.raises(ValueError):
        oracle.sparse_attn(at, np.array([[0, 4]], np.int32))


# --- IndexShare group ----------------------------------------------------------------

def _tiny_group(n_layers=4, same_indexer=False):
    wl = synth.WORKLOADS["tiny_l1k"].replace(T=80, S=80, k=16, schedule="F" * n_layers)
    layers = []
    for l in range(n_layers):
        layers.append(dict(ix=synth.indexer_inputs(wl, 0 if same_indexer else l),
                           at=synth.attn_inputs(wl, l)))
    return wl, layers


def test_group_shared_layers_reuse_full_layer_indices():
    wl, layers = _tiny_group()
    res = oracle.group_forward(layers, "FSSS", wl.k)
    f_idx = oracle.indexer_topk(layers[0]["ix"], wl.k)
    for l in range(4):
        assert np.array_equal(res[l]["idx"], f_idx)
        out, lse = oracle.sparse_attn(layers[l]["at"], f_idx)
        assert np.array_equal(res[l]["out"], out) and np.array_equal(res[l]["lse"], lse)
    # every shared layer has its own attention output
    assert not np.allclose(res[1]["out"], res[2]["out"])
    assert all(np.all(r["idx"] < np.arange(80)[:, None]) for r in res)  # causal: idx < t


def test_group_all_full_equals_independent_layers_and_fsss_with_equal_indexers():
    wl, layers = _tiny_group()
    ffff = oracle.group_forward(layers, "FFFF", wl.k)
    for l in range(4):
        idx = oracle.indexer_topk(layers[l]["ix"], wl.k)
        assert np.array_equal(ffff[l]["idx"], idx)
    wl, same = _tiny_group(same_indexer=True)
    a = oracle.group_forward(same, "FFFF", wl.k)
    b = oracle.group_forward(same, "FSSS", wl.k)
    for l in range(4):
        assert np.array_equal(a[l]["out"], b[l]["out"])
    _, mean = oracle.topk_overlap(a[0]["idx"], a[3]["idx"])
    assert mean == 1.0


def test_draft_steps_equal_an_fsss_walk_over_the_steps():
    """Draft-step reuse restated as an IndexShare schedule: the n draft steps are n layers of
    one query each, the first F (its indexer) and the rest S, all on the one shared cache; the
    stacked-query form must give the same positions and, step by step, the same outputs."""
    wl = synth.WORKLOADS["mtp_draft_b32_200k"].replace(B=3, S=300, q_pos0=300, k=24)
    layers = synth.group_inputs(wl, 4, with_indexer=True)
    walk = oracle.group_forward(layers, "FSSS", wl.k)
    at = dict(layers[0]["at"])
    at["q"] = torch.cat([l["at"]["q"] for l in layers], dim=1)  # [B, 4, H, DQK]
    idx, out, lse = oracle.draft_forward(layers[0]["ix"], at, wl.k)
    assert np.array_equal(idx, walk[0]["idx"])
    for s in range(4):
        assert np.array_equal(out[:, s], walk[s]["out"]) and np.array_equal(lse[:, s], walk[s]["lse"])
    # a subset of sequences gives those sequences' rows
    idx2, out2, _ = oracle.draft_forward(layers[0]["ix"], at, wl.k, seqs=[2, 0])
    assert np.array_equal(idx2, idx[[2, 0]]) and np.array_equal(out2, out[[2, 0]])
    # the steps keep their own queries: their outputs differ
    assert not np.allclose(out[:, 0], out[:, 1])


@pytest.mark.parametrize("bad", ["SFSS", "FSS", "FSSSF", "FSXS", ""])
def test_group_rejects_bad_schedules(bad):
    with pytest.raises(ValueError):
        oracle.check_schedule(bad, 4)


# --- overlap -------------------------------------------------------------------------

def test_overlap_brute_force_and_extremes():
    g = torch.Generator().manual_seed(21)
    R, k = 50, 32
    a = np.full((R, k), -1, np.int32)
    b = np.full((R, k), -1, np.int32)
    for r in range(R):
        na = int(torch.randint(0, k + 1, (1,), generator=g))
        a[r, :na] = np.sort(torch.randperm(100, generator=g)[:na].numpy())
        b[r, :na] = np.sort(torch.randperm(100, generator=g)[:na].numpy())
    per, mean = oracle.topk_overlap(a, b)
    for r in range(R):
        sa = set(a[r][a[r] >= 0].tolist())
        sb = set(b[r][b[r] >= 0].tolist())
        want = 1.0 if not sa else len(sa & sb) / len(sa)
        assert per[r] == pytest.approx(want, abs=0)
    assert mean == pytest.approx(per.mean(), rel=1e-12)
    assert oracle.topk_overlap(a, a)[1] == 1.0
    disj = np.arange(2 * k, dtype=np.int32).reshape(2, k)
    assert oracle.topk_overlap(disj[:1], disj[1:])[1] == 0.0


def _random_index_rows(g, R, k, universe, n_bufs):
    """n_bufs [R,k] buffers in top-k form; every buffer of a row has the same valid count
    (the same query sees the same keys in every layer)."""
    bufs = [np.full((R, k), -1, np.int32) for _ in range(n_bufs)]
    for r in range(R):
        nv = int(torch.randint(0, k + 1, (1,), generator=g))
        for b in bufs:
            b[r, :nv] = np.sort(torch.randperm(universe, generator=g)[:nv].numpy())
    return bufs


def test_overlap_matrix_brute_force_sets():
    g = torch.Generator().manual_seed(33)
    bufs = _random_index_rows(g, 40, 16, 40, 5)
    M, per = oracle.overlap_matrix(bufs)
    for i in range(5):
        for j in range(5):
            fr = []
            for r in range(40):
                si = set(bufs[i][r][bufs[i][r] >= 0].tolist())
                sj = set(bufs[j][r][bufs[j][r] >= 0].tolist())
                fr.append(1.0 if not si else len(si & sj) / len(si))
                assert per[r, i, j] == fr[-1]
            assert M[i, j] == pytest.approx(sum(fr) / len(fr), rel=1e-12)
    # equal valid counts per row make the matrix symmetric; every layer overlaps itself fully
    assert np.allclose(M, M.T, rtol=0, atol=1e-15)
    assert np.all(np.diag(M) == 1.0)


# A 4-layer overlap matrix worked by hand: layer 1 is close to 0, layer 3 to 2.
HAND_M = [[1.0, 0.9, 0.5, 0.2],
          [0.9, 1.0, 0.6, 0.3],
          [0.5, 0.6, 1.0, 0.7],
          [0.2, 0.3, 0.7, 1.0]]


@pytest.mark.parametrize("sched,want", [
    ("FSSS", (1.0 + 0.9 + 0.5 + 0.2) / 4),   # layers 1..3 reuse layer 0
    ("FSFS", (1.0 + 0.9 + 1.0 + 0.7) / 4),   # layer 1 reuses 0, layer 3 reuses 2
    ("FFSS", (1.0 + 1.0 + 0.6 + 0.3) / 4),   # layers 2, 3 reuse layer 1
    ("FSSF", (1.0 + 0.9 + 0.5 + 1.0) / 4),
    ("FFFF", 1.0),
])
def test_schedule_score_hand_worked(sched, want):
    assert oracle.schedule_score(HAND_M, sched) == pytest.approx(want, abs=1e-15)


def test_schedule_search_hand_worked():
    # two full layers: FSFS (0.9) beats FSSF (0.85), FFSS (0.725)
    best, arg = oracle.schedule_search(HAND_M, 2)
    assert arg == ["FSFS"] and best == pytest.approx(0.9, abs=1e-15)
    best, arg = oracle.schedule_search(HAND_M, 1)
    assert arg == ["FSSS"] and best == pytest.approx(0.65, abs=1e-15)
    best, arg = oracle.schedule_search(HAND_M, 4)
    assert arg == ["FFFF"] and best == 1.0
    # three full layers: FFFS (1+1+1+0.7)/4 = 0.925, FSFF (1+0.9+1+1)/4 = 0.975, FFSF 0.9
    best, arg = oracle.schedule_search(HAND_M, 3)
    assert arg == ["FSFF"] and best == pytest.approx(0.975, abs=1e-15)


# --- FP8 quantisation ----------------------------------------------------------------------

def _torch_e4m3(v):
    """torch's own fp32 -> e4m3fn conversion (round to nearest even) after clamping to the
    finite range: the library routine the encoder is pinned to."""
    t = torch.as_tensor(np.asarray(v, dtype=np.float32))
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_matches_torch_on_every_value_tie_and_range():
    finite = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    finite = finite[torch.isfinite(finite)].numpy().astype(np.float32)
    mags = np.unique(np.abs(finite))
    mids = ((mags[1:].astype(np.float64) + mags[:-1]) / 2).astype(np.float32)  # exact ties
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    g = np.random.default_rng(3)
    rand = (g.standard_normal(20000) * np.exp2(g.integers(-14, 10, 20000))).astype(np.float32)
    big = np.array([448.0, 449.0, 464.0, 465.0, 480.0, 1e6, 3.4e38], dtype=np.float32)
    tiny = np.array([2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 1e-30, 0.0], dtype=np.float32)
    v = np.concatenate([finite, mids, -mids, near, -near, rand, big, -big, tiny, -tiny])
    assert np.array_equal(oracle.encode_e4m3(v), _torch_e4m3(v))
    # round trip: every finite code decodes and re-encodes to itself
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.encode_e4m3(oracle.e4m3_to_double(codes)), codes)


def test_row_quantiser_matches_torch_ops():
    g = torch.Generator().manual_seed(8)
    rows, width = 64, 136
    x = torch.randn(rows, width, generator=g) * torch.exp2(torch.randint(-20, 12, (rows, 1), generator=g).float())
    x[5] = 0.0
    x[9, :] = 0.0
    x[9, 3] = -2.0 ** -30
    xb = x.to(torch.bfloat16)
    codes, scales = oracle.quantize_e4m3_rows(xb, width)
    xf = xb.float()
    amax = xf.abs().amax(-1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    want = (xf / sc[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales, sc.numpy())
    assert np.array_equal(codes, want)
    assert scales[5] == 1.0 and np.all(codes[5] == 0)
    # dequantised rows keep their largest magnitude: amax maps to the code of 448
    big = np.abs(xf.numpy()).argmax(1)
    assert np.all((codes[np.arange(rows), big] & 0x7F)[amax.numpy() > 0] == 0x7E)
