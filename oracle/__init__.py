"""Plain, slow, fp64 CPU oracle for the DSA hot path with IndexShare reuse.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` import this package.  It shares no code with the CUDA library
(``long_context_sparse_tcgen05_gb300``) and never imports it.

What it follows:
  * IndexShare explainer (sebastianraschka.com, llm-architecture-gallery/indexshare),
    "Why The Indexer Becomes Expensive": the indexer scores the preceding tokens of a
    query, the top-k positions are kept, main attention runs only on that subset.
  * same page, "How IndexShare Works": a full layer runs indexer + top-k and stores the
    positions; a shared layer skips both and uses the most recent full layer's positions.
  * IndexCache notes (digipro.cn/article/14223), section 2: the first layer is always F;
    S layers reuse the nearest preceding F layer's top-k.
  * GLM-5.2 IndexShare article, "What IndexShare reuses": the pattern is F,S,S,S and the
    shared layers keep their own queries, attention weights and outputs.
  * same article, "Reuse in the MTP layer": the first draft step of the multi-token-prediction
    layer computes the indices; the later draft steps reuse those indices and the KV cache.
  * The score formula I[t,s] = sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s]) is the project's
    statement of the indexer (the pages do not print one).
  * IndexCache notes, section 1: the indexer runs in FP8; its operands are e4m3 codes with one
    fp32 scale per token (the OCP E4M3 format, encoded and decoded here from its definition).

The numeric work sits in ``dsa_oracle.c`` (plain loops, double precision); this module
only marshals arrays and writes out the schedule walk.  Every function is pinned by
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, E4M3 = 0, 1

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP over rows).  Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_num_threads.restype = ctypes.c_int
            lib.orc_bf16_to_double.restype = ctypes.c_double
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_e4m3_to_double.restype = ctypes.c_double
            lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.orc_decode_bf16.argtypes = [_P, _P, _I64]
            lib.orc_decode_e4m3.argtypes = [_P, _P, _I64]
            lib.orc_visible.restype = _I64
            lib.orc_visible.argtypes = [_I64, _I64, _I64]
            lib.orc_indexer_scores.argtypes = [ctypes.c_int, _I64, ctypes.c_int, ctypes.c_int,
                                               _I64, _P, _P, _P, _P, _P, _P, _P, _I64, _P]
            lib.orc_topk_rows.argtypes = [_I64, _P, _I64, _P, ctypes.c_int, _P]
            lib.orc_sparse_attn.restype = _I64
            lib.orc_sparse_attn.argtypes = [_I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, _I64, _P, _P, _P, _I64, _P, _I64,
                                            _P, ctypes.c_int, _P, _P]
            lib.orc_encode_e4m3.restype = ctypes.c_uint8
            lib.orc_encode_e4m3.argtypes = [ctypes.c_float]
            lib.orc_encode_e4m3_array.argtypes = [_P, _P, _I64]
            lib.orc_quantize_e4m3_rows.argtypes = [_P, _I64, ctypes.c_int, _P, _P]
            lib.orc_topk_overlap.restype = ctypes.c_double
            lib.orc_topk_overlap.argtypes = [_P, _P, _I64, ctypes.c_int, _P]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().orc_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _raw(t, np_dtype):
    """Host bytes of a tensor (any device, any dtype) as a contiguous numpy array."""
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t).view(np_dtype)
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16, torch.int16):
        return t.view(torch.int16).numpy().view(np_dtype)
    if t.dtype in (torch.float8_e4m3fn, torch.uint8, torch.int8):
        return t.view(torch.uint8).numpy().view(np_dtype)
    return t.numpy().view(np_dtype)


def _rows(rows, n_total):
    if rows is None:
        return np.arange(n_total, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


# --- decoders -----------------------------------------------------------------------

def bf16_to_double(codes) -> np.ndarray:
    c = _raw(codes, np.uint16).reshape(-1)
    out = np.empty(c.size, dtype=np.float64)
    _load().orc_decode_bf16(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_to_double(codes) -> np.ndarray:
    c = _raw(codes, np.uint8).reshape(-1)
    out = np.empty(c.size, dtype=np.float64)
    _load().orc_decode_e4m3(_ptr(c), _ptr(out), c.size)
    return out


def encode_e4m3(values) -> np.ndarray:
    """E4M3 codes of fp32 values: nearest representable value, ties to even, saturated."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32).reshape(-1))
    out = np.empty(v.size, dtype=np.uint8)
    _load().orc_encode_e4m3_array(_ptr(v), _ptr(out), v.size)
    return out


def quantize_e4m3_rows(x, width: int):
    """(codes uint8 [rows, width], scales fp32 [rows]) of bf16 rows: scale = amax / 448 per
    row (1 for an all-zero row), code = e4m3(x / scale) in fp32."""
    c = _raw(x, np.uint16).reshape(-1, width)
    c = np.ascontiguousarray(c)
    codes = np.empty(c.shape, dtype=np.uint8)
    scales = np.empty(c.shape[0], dtype=np.float32)
    _load().orc_quantize_e4m3_rows(_ptr(c), c.shape[0], width, _ptr(codes), _ptr(scales))
    return codes, scales


def visible(S: int, q_pos: int, diag: int = 0) -> int:
    """Keys visible to a query at position q_pos: s < q_pos + diag, clipped to [0, S]."""
    return int(_load().orc_visible(S, q_pos, diag))


# --- indexer + top-k ----------------------------------------------------------------

def _dtype_code(t) -> int:
    if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
        return E4M3
    return BF16


def _take_rows(t, r: np.ndarray, flat_lead: int):
    """Rows r of a tensor whose first `flat_lead` dims are flattened (plain indexing)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(t)
    flat = t.reshape((-1,) + tuple(t.shape[flat_lead:]))
    return flat[torch.as_tensor(r, device=flat.device)].cpu()


def indexer_scores(ix: dict, rows=None) -> np.ndarray:
    """Scores [n_rows, S] (float64, -inf where not visible) of the given flat rows b*T+i.

    ``ix`` holds q [B,T,HI,DI], w [B,T,HI], k [B,S,DI] (bf16 or float8_e4m3fn), optional
    q_scale [B,T] / k_scale [B,S] fp32, q_pos0 (row i sits at position q_pos0 + i), diag."""
    k = ix["k"]
    S = k.shape[1]
    if "q_rows" in ix:  # operands already restricted to `rows` (flat ids over [B, T])
        qr, wr, qsr = ix["q_rows"], ix["w_rows"], ix.get("q_scale_rows")
        T, HI, DI = ix["T"], qr.shape[1], qr.shape[2]
        r = _rows(rows, 0)
    else:
        q, w, qs = ix["q"], ix["w"], ix.get("q_scale")
        B, T, HI, DI = q.shape
        r = _rows(rows, B * T)
        qr, wr = _take_rows(q, r, 2), _take_rows(w, r, 2)
        qsr = _take_rows(qs, r, 2) if qs is not None else None
    dt = _dtype_code(qr)
    npdt = np.uint8 if dt == E4M3 else np.uint16
    qa = _raw(qr, npdt)
    ka = _raw(k, npdt)
    wa = _raw(wr.float(), np.float32)
    ks = ix.get("k_scale")
    qsa = _raw(qsr.float(), np.float32) if qsr is not None else None
    ksa = _raw(ks.float(), np.float32) if ks is not None else None
    rb = np.ascontiguousarray(r // T)
    rp = np.ascontiguousarray(r % T + int(ix.get("q_pos0", 0)))
    out = np.empty((r.size, S), dtype=np.float64)
    _load().orc_indexer_scores(dt, S, HI, DI, r.size, _ptr(qa),
                               _ptr(qsa) if qsa is not None else None, _ptr(wa), _ptr(rb),
                               _ptr(rp), _ptr(ka), _ptr(ksa) if ksa is not None else None,
                               int(ix.get("diag", 0)), _ptr(out))
    return out


def topk_rows(scores: np.ndarray, n_valid, k: int) -> np.ndarray:
    """Top-k [R, k] int32 of each score row under (score desc, position asc), ascending
    positions, -1 padded.  Only the first n_valid[r] entries of row r are candidates."""
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64))
    if s.ndim == 1:
        s = s[None]
    R, ld = s.shape
    nv = np.ascontiguousarray(np.broadcast_to(np.asarray(n_valid, dtype=np.int64), (R,)))
    idx = np.empty((R, k), dtype=np.int32)
    _load().orc_topk_rows(R, _ptr(s), ld, _ptr(nv), int(k), _ptr(idx))
    return idx


def row_visible(ix_or_shape: dict, rows) -> np.ndarray:
    """Visible-key count of each flat row b*T+i."""
    T = ix_or_shape["T"] if "T" in ix_or_shape else ix_or_shape["q"].shape[1]
    if "q_rows" in ix_or_shape:
        T = ix_or_shape["T"]
    S = ix_or_shape["S"] if "S" in ix_or_shape else ix_or_shape["k"].shape[1]
    q_pos0 = int(ix_or_shape.get("q_pos0", 0))
    diag = int(ix_or_shape.get("diag", 0))
    r = np.asarray(rows, dtype=np.int64)
    n = (r % T) + q_pos0 + diag
    return np.clip(n, 0, S)


def indexer_topk(ix: dict, k: int, rows=None, return_scores: bool = False):
    """Index rows [n_rows, k] of a full (F) layer: scores, then top-k."""
    r = _rows(rows, ix["q"].shape[0] * ix["q"].shape[1]) if "q" in ix else _rows(rows, 0)
    sc = indexer_scores(ix, r)
    idx = topk_rows(sc, row_visible(ix, r), k)
    return (idx, sc) if return_scores else idx


# --- sparse attention ---------------------------------------------------------------

def sparse_attn(at: dict, idx_rows, rows=None):
    """(out [n_rows,H,DV], lse [n_rows,H]) in float64 for the given flat rows b*T+i.

    ``at`` holds q [B,T,H,DQK] bf16, k [B,S,>=DQK] bf16, optional v [B,S,>=DV] bf16
    (absent: v is k, the latent-KV form), d_v, scale.  ``idx_rows`` is [n_rows, kk]."""
    k = at["k"]
    v = at.get("v")
    S, k_ld = k.shape[1], k.shape[2]
    DV = int(at["d_v"])
    if "q_rows" in at:  # queries already restricted to `rows`
        qr, T = at["q_rows"], at["T"]
        r = _rows(rows, 0)
    else:
        B, T = at["q"].shape[:2]
        r = _rows(rows, B * T)
        qr = _take_rows(at["q"], r, 2)
    H, DQK = qr.shape[1], qr.shape[2]
    qa = _raw(qr, np.uint16)
    ka = _raw(k, np.uint16)
    if v is None:
        va, v_ld = ka, k_ld
    else:
        va, v_ld = _raw(v, np.uint16), v.shape[2]
    ir = np.ascontiguousarray(np.asarray(idx_rows, dtype=np.int32))
    assert ir.shape[0] == r.size
    kk = ir.shape[1]
    rb = np.ascontiguousarray(r // T)
    out = np.empty((r.size, H, DV), dtype=np.float64)
    lse = np.empty((r.size, H), dtype=np.float64)
    bad = _load().orc_sparse_attn(S, H, DQK, DV, float(at["scale"]), r.size, _ptr(qa), _ptr(rb),
                                  _ptr(ka), k_ld, _ptr(va), v_ld, _ptr(ir), kk, _ptr(out),
                                  _ptr(lse))
    if bad:
        raise ValueError(f"{bad} index entries outside [-1, S)")
    return out, lse


# --- IndexShare group ---------------------------------------------------------------

def check_schedule(schedule: str, n_layers: int) -> None:
    """A schedule has one 'F' (full) or 'S' (shared) per layer and starts with 'F'."""
    if len(schedule) != n_layers or not schedule or schedule[0] != "F" or set(schedule) - {"F", "S"}:
        raise ValueError(f"bad schedule {schedule!r} for {n_layers} layers")


def group_forward(layers, schedule: str, k: int, rows=None):
    """Walk an F/S schedule.  An F layer runs indexer + top-k and keeps the positions; an S
    layer reuses the most recent F layer's positions.  Every layer runs its own attention
    with its own Q/KV.  Returns one dict(idx, out, lse) per layer."""
    check_schedule(schedule, len(layers))
    cur = None
    res = []
    for layer, role in zip(layers, schedule):
        if role == "F":
            cur = indexer_topk(layer["ix"], k, rows)
        out, lse = sparse_attn(layer["at"], cur, rows)
        res.append(dict(idx=cur, out=out, lse=lse))
    return res


def draft_forward(ix: dict, at: dict, k: int, seqs=None):
    """Draft steps of a multi-token-prediction layer: the first step's indexer + top-k picks
    each sequence's positions (``ix``: one query per sequence), then every draft step s of
    sequence b (``at["q"]`` [B, n, H, DQK], one shared KV) attends over those positions.
    Returns (idx [m, k], out [m, n, H, DV], lse [m, n, H]) for the m sequences ``seqs``."""
    B, n = at["q"].shape[:2]
    seqs = list(range(B)) if seqs is None else [int(b) for b in seqs]
    idx = indexer_topk(ix, k, seqs)  # flat row b*1 + 0 of the one-query indexer
    rows = [b * n + s for b in seqs for s in range(n)]
    out, lse = sparse_attn(at, np.repeat(idx, n, axis=0), rows)
    return idx, out.reshape(len(seqs), n, *out.shape[1:]), lse.reshape(len(seqs), n, lse.shape[1])


# --- overlap ------------------------------------------------------------------------

def topk_overlap(a, b):
    """(per_row, mean): |A and B| / |A| over valid entries, per row."""
    aa = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    bb = np.ascontiguousarray(np.asarray(b, dtype=np.int32))
    assert aa.shape == bb.shape
    k = aa.shape[-1]
    aa = aa.reshape(-1, k)
    bb = bb.reshape(-1, k)
    per = np.empty(aa.shape[0], dtype=np.float64)
    mean = _load().orc_topk_overlap(_ptr(aa), _ptr(bb), aa.shape[0], k, _ptr(per))
    return per, float(mean)


def overlap_matrix(bufs):
    """M[i][j] = topk_overlap(bufs[i], bufs[j]) mean, for every ordered pair of n index
    buffers over the same rows (the pairwise-overlap heatmap of the IndexCache notes,
    section 2), plus the per-row fractions [rows, n, n]."""
    n = len(bufs)
    M = np.ones((n, n), dtype=np.float64)
    per = None
    for i in range(n):
        for j in range(n):
            pr, m = topk_overlap(bufs[i], bufs[j])
            if per is None:
                per = np.empty((pr.shape[0], n, n), dtype=np.float64)
            per[:, i, j] = pr
            M[i, j] = m
    return M, per


def schedule_score(M, schedule: str) -> float:
    """A shared layer reuses the most recent full layer's positions (explainer, "How
    IndexShare Works"), so it keeps the fraction M[l][f] of its own top-k, f being that full
    layer; a full layer keeps all of it.  The score is the mean of that over the layers."""
    M = np.asarray(M, dtype=np.float64)
    check_schedule(schedule, M.shape[0])
    total = 0.0
    f = 0
    for l, role in enumerate(schedule):
        if role == "F":
            f = l
        total += M[l, f]
    return total / M.shape[0]


def schedule_search(M, n_full: int):
    """(best score, every schedule reaching it) over all schedules with n_full full layers,
    the first layer among them: plain enumeration."""
    import itertools
    n = np.asarray(M).shape[0]
    best, arg = None, []
    for rest in itertools.combinations(range(1, n), n_full - 1):
        sched = "".join("F" if (l == 0 or l in rest) else "S" for l in range(n))
        v = schedule_score(M, sched)
        if best is None or v > best + 1e-12:
            best, arg = v, [sched]
        elif abs(v - best) <= 1e-12:
            arg.append(sched)
    return best, arg
