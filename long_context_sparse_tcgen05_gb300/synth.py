"""Seeded synthetic inputs for the DSA + IndexShare hot path.

This module only draws random tensors and packs them into the operand layouts of the
library; it holds none of the method's arithmetic, and both the CUDA path and the CPU
oracle consume exactly the bytes it produces.  The shapes and value distributions follow
the workloads the project is measured on:

* ``tiny_l1k``           1 sequence, L=1,024, indexer H_I=4, d_I=64 on small integers,
                         k=64, four layers F,S,S,S of 8-head MQA attention, d=64.
* ``prefill_16k``        1 sequence, L=16,384, bf16 N(0,1) indexer H_I=64, d_I=128, k=2,048,
                         four layers F,S,S,S of 64-head sparse MQA over a 576-dim latent KV.
* ``prefill_128k``       1 sequence, L=131,072, FP8 e4m3 indexer with per-token scales,
                         inputs correlated across layers, 8 layers (two F,S,S,S groups).
* ``decode_b32_200k``    32 sequences x 1 new query over a 200,000-token cache, FP8 indexer,
                         16 layers (four F,S,S,S groups).
* ``chunked_prefill_1m`` the last 4,096 rows of a 1,048,576-token sequence against the full
                         causal cache, FP8 indexer, correlated inputs, 16 layers.
* ``heatmap_128k``       the 128K shapes over 16 layers run all-F, for the layer-overlap
                         heatmap: indexer inputs correlated in clusters of layers.
* ``mtp_draft_b32_200k`` four draft steps of a multi-token-prediction layer over the 32 x
                         200,000-token decode cache: every step has its own queries, all share
                         the layer's caches (indexer keys and latent KV) and see the same keys.

Every tensor is drawn from its own Philox stream, seeded by
``20261202 + 1000*workload_id + 10*layer + tensor_id``; tensors longer than one chunk are
drawn chunk by chunk along the token axis (each chunk re-seeded from the tensor seed and
the chunk number), so a row's values do not depend on how much of the tensor is made.
FP8 operands are produced by per-token quantisation: scale = amax/448 over the token's
features, code = round-to-nearest-even(x/scale) saturated to +-448 (torch's e4m3 cast).
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED_BASE = 20261202
CHUNK = 4096  # tokens per independently seeded chunk

T_Q_I, T_K_I, T_W, T_Q, T_KV, T_V = 0, 1, 2, 3, 4, 5
T_BASE_Q_I, T_BASE_K_I = 7, 8
T_CLUSTER_Q_I, T_CLUSTER_K_I = 6, 9  # drawn per cluster (the cluster id takes the layer slot)
CLUSTER_SHARE = 0.75                 # share of a layer's noise variance common to its cluster


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int            # workload id used in the seeds
    B: int              # sequences
    T: int              # query rows per sequence
    S: int              # keys per sequence
    q_pos0: int         # absolute position of query row 0
    HI: int             # indexer heads
    DI: int             # indexer head dim
    idx_dtype: str      # "bf16" | "e4m3"
    values: str         # "int" | "gauss" | "correlated"
    k: int              # top-k
    schedule: str       # one 'F'/'S' per layer
    H: int              # attention query heads
    DQK: int            # q/k head dim (latent + rope for MLA)
    DV: int             # value dim
    latent: bool        # True: V is the first DV columns of the KV row (one buffer)
    diag: int = 0       # keys s < q_pos + diag are visible
    clusters: tuple = ()  # "clustered" values: cluster id of each layer
    shared_cache: bool = False  # every "layer" (draft step) reads layer 0's keys and KV

    @property
    def n_layers(self) -> int:
        return len(self.schedule)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.DQK)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_l1k": Workload("tiny_l1k", 0, 1, 1024, 1024, 0, 4, 64, "bf16", "int", 64, "FSSS",
                         8, 64, 64, False),
    "prefill_16k": Workload("prefill_16k", 1, 1, 16384, 16384, 0, 64, 128, "bf16", "gauss",
                            2048, "FSSS", 64, 576, 512, True),
    "prefill_128k": Workload("prefill_128k", 2, 1, 131072, 131072, 0, 64, 128, "e4m3",
                             "correlated", 2048, "FSSSFSSS", 64, 576, 512, True),
    "decode_b32_200k": Workload("decode_b32_200k", 3, 32, 1, 200000, 200000, 64, 128, "e4m3",
                                "gauss", 2048, "FSSS" * 4, 64, 576, 512, True),
    "chunked_prefill_1m": Workload("chunked_prefill_1m", 4, 1, 4096, 1048576, 1048576 - 4096,
                                   64, 128, "e4m3", "correlated", 2048, "FSSS" * 4, 64, 576, 512,
                                   True),
    "mtp_draft_b32_200k": Workload("mtp_draft_b32_200k", 6, 32, 1, 200000, 200000, 64, 128, "e4m3",
                                   "gauss", 2048, "FSSS", 64, 576, 512, True, shared_cache=True),
    "heatmap_128k": Workload("heatmap_128k", 5, 1, 131072, 131072, 0, 64, 128, "e4m3", "clustered",
                             2048, "F" * 16, 64, 576, 512, True,
                             clusters=(0, 1, 1, 2, 2, 2, 3, 3, 3, 3, 3, 3, 3, 3, 3, 3)),
}


def seed_of(wl: Workload, layer: int, tensor_id: int) -> int:
    return SEED_BASE + 1000 * wl.wid + 10 * layer + tensor_id


def _cache_layer(wl: Workload, layer: int) -> int:
    """Layer whose seeds draw this layer's keys and KV (layer 0 for a shared cache)."""
    return 0 if wl.shared_cache else layer


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _draw_chunk(kind, sub, device, seed, chunk, lo, hi):
    g = _gen(device, seed * 1000003 + chunk)
    if kind == "normal":
        return torch.randn(sub, generator=g, device=device)
    if kind == "uniform":
        return torch.rand(sub, generator=g, device=device)
    if kind == "int":
        return torch.randint(lo, hi + 1, sub, generator=g, device=device).float()
    raise ValueError(kind)


def _draw(kind: str, shape, device, seed: int, lo: int = 0, hi: int = 0) -> torch.Tensor:
    """fp32 tensor of `shape`, drawn chunk by chunk along dim 1 (the token axis)."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    n = shape[1]
    for c0 in range(0, n, CHUNK):
        c1 = min(n, c0 + CHUNK)
        sub = (shape[0], c1 - c0) + tuple(shape[2:])
        out[:, c0:c1] = _draw_chunk(kind, sub, device, seed, c0 // CHUNK, lo, hi)
    return out


def _draw_rows(kind: str, shape, device, seed: int, flat_rows, lo: int = 0, hi: int = 0):
    """Rows (flat b*shape[1] + t) of the tensor _draw would make, drawing only the chunks
    that hold them (chunks are seeded independently, so the values are identical)."""
    n = shape[1]
    out = torch.empty((len(flat_rows),) + tuple(shape[2:]), dtype=torch.float32, device=device)
    cache = {}
    for i, r in enumerate(flat_rows):
        t = r % n
        c = t // CHUNK
        if c not in cache:
            c0, c1 = c * CHUNK, min(n, (c + 1) * CHUNK)
            cache[c] = _draw_chunk(kind, (shape[0], c1 - c0) + tuple(shape[2:]), device, seed, c, lo, hi)
        out[i] = cache[c][r // n, t - c * CHUNK]
    return out


def quantize_e4m3_per_token(x: torch.Tensor, token_dims: int):
    """(codes, scale): one fp32 scale per token (the first `token_dims` dims of x)."""
    flat = x.reshape(x.shape[:token_dims] + (-1,))
    amax = flat.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    y = x / scale.reshape(scale.shape + (1,) * (x.dim() - token_dims))
    return y.clamp(-448.0, 448.0).to(torch.float8_e4m3fn), scale.float().contiguous()


def indexer_inputs(wl: Workload, layer: int, device="cpu") -> dict:
    """Indexer operands of one layer: q [B,T,HI,DI], w [B,T,HI], k [B,S,DI] (+ scales)."""
    qs = (wl.B, wl.T, wl.HI, wl.DI)
    ks = (wl.B, wl.S, wl.DI)
    ws = (wl.B, wl.T, wl.HI)
    if wl.values == "int":
        q = _draw("int", qs, device, seed_of(wl, layer, T_Q_I), -3, 3)
        k = _draw("int", ks, device, seed_of(wl, _cache_layer(wl, layer), T_K_I), -3, 3)
        w = _draw("int", ws, device, seed_of(wl, layer, T_W), 1, 4)
    elif wl.values == "gauss":
        q = _draw("normal", qs, device, seed_of(wl, layer, T_Q_I))
        k = _draw("normal", ks, device, seed_of(wl, _cache_layer(wl, layer), T_K_I))
        w = _draw("uniform", ws, device, seed_of(wl, layer, T_W)) / 8.0
    elif wl.values == "correlated":
        # shared base + 0.3 * independent per-layer noise; w is drawn once for all layers
        q = _draw("normal", qs, device, seed_of(wl, 0, T_BASE_Q_I))
        q += 0.3 * _draw("normal", qs, device, seed_of(wl, layer, T_Q_I))
        k = _draw("normal", ks, device, seed_of(wl, 0, T_BASE_K_I))
        k += 0.3 * _draw("normal", ks, device, seed_of(wl, _cache_layer(wl, layer), T_K_I))
        w = _draw("uniform", ws, device, seed_of(wl, 0, T_W)) / 8.0
    elif wl.values == "clustered":
        # shared base + 0.3 * (unit-variance noise), the noise mixing a component drawn once
        # per cluster of layers with the layer's own: each layer's values are distributed as
        # in "correlated", and layers of one cluster share CLUSTER_SHARE of their noise
        a, b = math.sqrt(CLUSTER_SHARE), math.sqrt(1.0 - CLUSTER_SHARE)
        c = wl.clusters[layer]
        q = _draw("normal", qs, device, seed_of(wl, 0, T_BASE_Q_I))
        q += (0.3 * a) * _draw("normal", qs, device, seed_of(wl, c, T_CLUSTER_Q_I))
        q += (0.3 * b) * _draw("normal", qs, device, seed_of(wl, layer, T_Q_I))
        k = _draw("normal", ks, device, seed_of(wl, 0, T_BASE_K_I))
        k += (0.3 * a) * _draw("normal", ks, device, seed_of(wl, c, T_CLUSTER_K_I))
        k += (0.3 * b) * _draw("normal", ks, device, seed_of(wl, _cache_layer(wl, layer), T_K_I))
        w = _draw("uniform", ws, device, seed_of(wl, 0, T_W)) / 8.0
    else:
        raise ValueError(wl.values)
    ix = dict(w=w.contiguous(), q_pos0=wl.q_pos0, diag=wl.diag)
    if wl.idx_dtype == "bf16":
        ix["q"] = q.to(torch.bfloat16).contiguous()
        ix["k"] = k.to(torch.bfloat16).contiguous()
        ix["q_scale"] = None
        ix["k_scale"] = None
    elif wl.values == "int":
        # small integers are exact e4m3 codes: unit scales
        ix["q"] = q.to(torch.float8_e4m3fn).contiguous()
        ix["k"] = k.to(torch.float8_e4m3fn).contiguous()
        ix["q_scale"] = torch.ones((wl.B, wl.T), dtype=torch.float32, device=device)
        ix["k_scale"] = torch.ones((wl.B, wl.S), dtype=torch.float32, device=device)
    else:
        ix["q"], ix["q_scale"] = quantize_e4m3_per_token(q, 2)
        ix["k"], ix["k_scale"] = quantize_e4m3_per_token(k, 2)
    del q, k
    return ix


def attn_inputs(wl: Workload, layer: int, device="cpu", kv_of=None) -> dict:
    """Attention operands of one layer: q [B,T,H,DQK] bf16 and either a latent KV
    [B,S,DQK] (V = its first DV columns) or separate K [B,S,DQK] and V [B,S,DV].  kv_of: an
    attention dict whose KV tensors this layer shares (a shared cache) instead of drawing."""
    q = _draw("normal", (wl.B, wl.T, wl.H, wl.DQK), device, seed_of(wl, layer, T_Q))
    at = dict(q=q.to(torch.bfloat16).contiguous(), d_v=wl.DV, scale=wl.scale)
    del q
    if kv_of is not None:
        at["k"], at["v"] = kv_of["k"], kv_of["v"]
        return at
    kv = _draw("normal", (wl.B, wl.S, wl.DQK), device, seed_of(wl, _cache_layer(wl, layer), T_KV))
    at["k"] = kv.to(torch.bfloat16).contiguous()
    del kv
    if wl.latent:
        at["v"] = None
    else:
        v = _draw("normal", (wl.B, wl.S, wl.DV), device, seed_of(wl, _cache_layer(wl, layer), T_V))
        at["v"] = v.to(torch.bfloat16).contiguous()
    return at


def indexer_rows(wl: Workload, layer: int, rows, device="cpu") -> dict:
    """Indexer operands with only the given query rows drawn: q_rows [n,HI,DI], w_rows,
    q_scale_rows, plus the full keys; identical values to indexer_inputs at those rows."""
    assert wl.values in ("gauss", "correlated", "clustered"), "row subsets are for the Gaussian workloads"
    qs = (wl.B, wl.T, wl.HI, wl.DI)
    ws = (wl.B, wl.T, wl.HI)
    full = indexer_inputs(wl.replace(T=1, q_pos0=0), layer, device)  # keys only matter here
    if wl.values == "gauss":
        q = _draw_rows("normal", qs, device, seed_of(wl, layer, T_Q_I), rows)
        w = _draw_rows("uniform", ws, device, seed_of(wl, layer, T_W), rows) / 8.0
    elif wl.values == "correlated":
        q = _draw_rows("normal", qs, device, seed_of(wl, 0, T_BASE_Q_I), rows)
        q += 0.3 * _draw_rows("normal", qs, device, seed_of(wl, layer, T_Q_I), rows)
        w = _draw_rows("uniform", ws, device, seed_of(wl, 0, T_W), rows) / 8.0
    else:
        a, b = math.sqrt(CLUSTER_SHARE), math.sqrt(1.0 - CLUSTER_SHARE)
        c = wl.clusters[layer]
        q = _draw_rows("normal", qs, device, seed_of(wl, 0, T_BASE_Q_I), rows)
        q += (0.3 * a) * _draw_rows("normal", qs, device, seed_of(wl, c, T_CLUSTER_Q_I), rows)
        q += (0.3 * b) * _draw_rows("normal", qs, device, seed_of(wl, layer, T_Q_I), rows)
        w = _draw_rows("uniform", ws, device, seed_of(wl, 0, T_W), rows) / 8.0
    ix = dict(k=full["k"], k_scale=full["k_scale"], w_rows=w.contiguous(), T=wl.T, S=wl.S,
              q_pos0=wl.q_pos0, diag=wl.diag, B=wl.B)
    if wl.idx_dtype == "bf16":
        ix["q_rows"], ix["q_scale_rows"] = q.to(torch.bfloat16).contiguous(), None
    else:
        ix["q_rows"], ix["q_scale_rows"] = quantize_e4m3_per_token(q, 1)
    return ix


def attn_rows(wl: Workload, layer: int, rows, device="cpu") -> dict:
    """Attention operands with only the given query rows drawn (q_rows [n,H,DQK]) plus the
    full KV; identical values to attn_inputs at those rows."""
    q = _draw_rows("normal", (wl.B, wl.T, wl.H, wl.DQK), device, seed_of(wl, layer, T_Q), rows)
    at = dict(q_rows=q.to(torch.bfloat16).contiguous(), d_v=wl.DV, scale=wl.scale, T=wl.T)
    kv = _draw("normal", (wl.B, wl.S, wl.DQK), device, seed_of(wl, _cache_layer(wl, layer), T_KV))
    at["k"] = kv.to(torch.bfloat16).contiguous()
    at["v"] = None
    if not wl.latent:
        v = _draw("normal", (wl.B, wl.S, wl.DV), device, seed_of(wl, _cache_layer(wl, layer), T_V))
        at["v"] = v.to(torch.bfloat16)
    return at


def group_inputs(wl: Workload, n_layers: int, device="cpu", with_indexer=None) -> list:
    """layer_inputs of layers 0 .. n_layers-1; with a shared cache the key and KV tensors of
    layer 0 are reused by every layer (the values are identical; they are drawn once)."""
    out = []
    for l in range(n_layers):
        if not wl.shared_cache or l == 0:
            out.append(layer_inputs(wl, l, device, with_indexer))
            continue
        need_ix = wl.schedule[l] == "F" if with_indexer is None else with_indexer
        ix = None
        if need_ix:
            ix = indexer_inputs(wl.replace(S=1), l, device)  # this step's queries only
            src = out[0]["ix"] if out[0]["ix"] is not None else indexer_inputs(wl, 0, device)
            ix["k"], ix["k_scale"] = src["k"], src["k_scale"]
        out.append(dict(ix=ix, at=attn_inputs(wl, l, device, kv_of=out[0]["at"])))
    return out


def layer_inputs(wl: Workload, layer: int, device="cpu", with_indexer=None) -> dict:
    """One layer's operands; indexer inputs only for F layers unless asked otherwise."""
    need_ix = wl.schedule[layer] == "F" if with_indexer is None else with_indexer
    return dict(ix=indexer_inputs(wl, layer, device) if need_ix else None,
                at=attn_inputs(wl, layer, device))


def scores_input(R: int, n: int, device="cpu", kind: str = "normal", seed: int = 7,
                 lo: int = -2, hi: int = 2) -> torch.Tensor:
    """fp32 score rows [R, n] for exercising a standalone top-k."""
    if kind == "normal":
        return _draw("normal", (1, R, n), device, SEED_BASE + seed)[0]
    return _draw("int", (1, R, n), device, SEED_BASE + seed, lo, hi)[0]


def sample_rows(wl: Workload, n: int, seed: int = 11) -> list:
    """Flat row ids b*T+i to check: the first rows (fewer than k keys visible), the last
    rows, and uniformly random rows in between."""
    total = wl.B * wl.T
    if total <= n:
        return list(range(total))
    g = torch.Generator().manual_seed(SEED_BASE + seed)
    head = list(range(min(4, total)))
    tail = list(range(max(0, total - 4), total))
    first_full = [i for i in (wl.k - wl.q_pos0 - wl.diag - 1, wl.k - wl.q_pos0 - wl.diag)
                  if 0 <= i < wl.T]
    rest = torch.randint(0, total, (n,), generator=g).tolist()
    return sorted(set(head + tail + first_full + rest))
