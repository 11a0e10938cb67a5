"""DeepSeek Sparse Attention with IndexShare reuse on one GB300 (sm_103a).

Thin ctypes binding over ``libdsa.so`` (C ABI in ``include/dsa.h``).  The functions here
only marshal torch tensors into the C structs (device pointers, sizes, the current CUDA
stream) and allocate outputs; every step of the computation runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing the first call raises.

Calls (same names as the C ABI):
  indexer_scores(ix)                      -> fp32 scores [B,T,S]
  dsa_topk(k, ix=... | scores=...)        -> int32 idx [B,T,k]
  dsa_sparse_attn(at, idx)                -> (out [B,T,H,d_v] bf16, lse [B,T,H] fp32)
  indexshare_group_forward(layers, schedule, k) -> (outs, lses, idx_bufs)
  indexshare_group_forward_varlen(layers, schedule, k, cu_q, cu_k, q_pos0) -> same, packed rows
  indexshare_draft_forward(ix, at, k)     -> (out [B,n,H,d_v], lse [B,n,H], idx [B,1,k]): n draft
                                             steps over the first step's selection, one launch
  topk_overlap(a, b)                      -> (per_row fp32, mean float)
  topk_overlap_matrix(bufs)               -> (n x n mean overlaps, counts [rows,n,n] or None)
  indexshare_schedule_score(M, schedule)  -> float (host only)
  indexshare_schedule_search(M, n_full)   -> (schedule str, score) (host only)
  dsa_quantize_e4m3_append(x, codes, scales, pos0 | positions) -> e4m3 rows + scales in a cache
Operand dicts use the keys produced by ``synth``: an indexer dict holds q, w, k, q_scale,
k_scale, q_pos0, diag; an attention dict holds q, k, v (None: latent KV), d_v, scale.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_BF16, DSA_E4M3 = 0, 1
TOPK_FROM_SCORES, TOPK_FROM_INDEXER = 0, 1
FLAG_BAD_INDEX, FLAG_NAN_SCORE, FLAG_UNSORTED, FLAG_TIMEOUT = 0x1, 0x2, 0x4, 0x8
WS_MIN = 256

_c = ctypes
_P = _c.c_void_p


class IndexerArgs(_c.Structure):
    _fields_ = [("B", _c.c_int32), ("T", _c.c_int32), ("S", _c.c_int32), ("H_I", _c.c_int32),
                ("d_I", _c.c_int32), ("dtype", _c.c_int), ("q", _P), ("q_scale", _P), ("w", _P),
                ("k", _P), ("k_scale", _P), ("q_pos0", _c.c_int64), ("diag", _c.c_int32),
                ("q_stride_b", _c.c_int64), ("q_stride_t", _c.c_int64), ("k_stride_b", _c.c_int64)]


class AttnArgs(_c.Structure):
    _fields_ = [("B", _c.c_int32), ("T", _c.c_int32), ("S", _c.c_int32), ("H", _c.c_int32),
                ("d_qk", _c.c_int32), ("d_v", _c.c_int32), ("scale", _c.c_float), ("q", _P),
                ("k", _P), ("k_ld", _c.c_int64), ("v", _P), ("v_ld", _c.c_int64),
                ("q_stride_b", _c.c_int64), ("q_stride_t", _c.c_int64), ("k_stride_b", _c.c_int64),
                ("v_stride_b", _c.c_int64)]


class TopkSrc(_c.Structure):
    _fields_ = [("kind", _c.c_int), ("scores", _P), ("ld", _c.c_int64),
                ("ix", _c.POINTER(IndexerArgs))]


class Layer(_c.Structure):
    _fields_ = [("ix", IndexerArgs), ("at", AttnArgs), ("out", _P), ("lse", _P)]


class Varlen(_c.Structure):
    _fields_ = [("n_seqs", _c.c_int32), ("cu_q", _c.POINTER(_c.c_int64)), ("cu_k", _c.POINTER(_c.c_int64)),
                ("q_pos0", _c.POINTER(_c.c_int64))]


class DsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_string(status)}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libdsa.so (built by ``build.build()``).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libdsa.so not found at {path}: run "
                                   "long_context_sparse_tcgen05_gb300.build.build() first")
            lib = _c.CDLL(path)
            S = _c.c_int
            lib.dsa_workspace_size.restype = _c.c_size_t
            lib.dsa_workspace_size.argtypes = [_c.POINTER(IndexerArgs), _c.c_int32]
            lib.dsa_topk_workspace_size.restype = _c.c_size_t
            lib.dsa_topk_workspace_size.argtypes = [_c.c_int32, _c.c_int32, _c.c_int32, _c.c_int64, _c.c_int32,
                                                    _c.c_int32]
            lib.dsa_attn_workspace_size.restype = _c.c_size_t
            lib.dsa_attn_workspace_size.argtypes = [_c.POINTER(AttnArgs), _c.c_int32]
            lib.indexshare_group_workspace_size.restype = _c.c_size_t
            lib.indexshare_group_workspace_size.argtypes = [_c.POINTER(Layer), _c.c_int32, _c.c_char_p, _c.c_int32,
                                                            _c.POINTER(Varlen)]
            lib.dsa_set_wait_limit.restype = None
            lib.dsa_set_wait_limit.argtypes = [_c.c_uint64]
            lib.dsa_indexer_scores.restype = S
            lib.dsa_indexer_scores.argtypes = [_c.POINTER(IndexerArgs), _P, _c.c_int64, _P,
                                               _c.c_size_t, _P]
            lib.dsa_topk.restype = S
            lib.dsa_topk.argtypes = [_c.POINTER(TopkSrc), _c.c_int32, _c.c_int32, _c.c_int32,
                                     _c.c_int64, _c.c_int32, _c.c_int32, _P, _P, _c.c_size_t, _P]
            lib.dsa_sparse_attn.restype = S
            lib.dsa_sparse_attn.argtypes = [_c.POINTER(AttnArgs), _P, _c.c_int32, _P, _P, _P,
                                            _c.c_size_t, _P]
            lib.indexshare_group_forward.restype = S
            lib.indexshare_group_forward.argtypes = [_c.POINTER(Layer), _c.c_int32, _c.c_char_p,
                                                     _c.c_int32, _c.POINTER(_P), _P, _c.c_size_t,
                                                     _P]
            lib.indexshare_draft_forward.restype = S
            lib.indexshare_draft_forward.argtypes = [_c.POINTER(IndexerArgs), _c.POINTER(AttnArgs), _c.c_int32,
                                                     _P, _P, _P, _P, _c.c_size_t, _P]
            lib.indexshare_draft_workspace_size.restype = _c.c_size_t
            lib.indexshare_draft_workspace_size.argtypes = [_c.POINTER(IndexerArgs), _c.POINTER(AttnArgs),
                                                            _c.c_int32]
            lib.indexshare_group_forward_varlen.restype = S
            lib.indexshare_group_forward_varlen.argtypes = [_c.POINTER(Layer), _c.c_int32, _c.c_char_p, _c.c_int32,
                                                            _c.POINTER(Varlen), _c.POINTER(_P), _P, _c.c_size_t, _P]
            lib.dsa_workspace_size_varlen.restype = _c.c_size_t
            lib.dsa_workspace_size_varlen.argtypes = [_c.POINTER(IndexerArgs), _c.POINTER(Varlen), _c.c_int32]
            lib.topk_overlap.restype = S
            lib.topk_overlap.argtypes = [_P, _P, _c.c_int32, _c.c_int32, _P,
                                         _c.POINTER(_c.c_double), _P, _c.c_size_t, _P]
            lib.topk_overlap_matrix.restype = S
            lib.topk_overlap_matrix.argtypes = [_c.POINTER(_P), _c.c_int32, _c.c_int32, _c.c_int32, _P,
                                                _c.POINTER(_c.c_double), _P, _c.c_size_t, _P]
            lib.topk_overlap_matrix_workspace_size.restype = _c.c_size_t
            lib.topk_overlap_matrix_workspace_size.argtypes = [_c.c_int32]
            lib.indexshare_schedule_score.restype = S
            lib.indexshare_schedule_score.argtypes = [_c.POINTER(_c.c_double), _c.c_int32, _c.c_char_p,
                                                      _c.POINTER(_c.c_double)]
            lib.indexshare_schedule_search.restype = S
            lib.indexshare_schedule_search.argtypes = [_c.POINTER(_c.c_double), _c.c_int32, _c.c_int32,
                                                       _c.c_char_p, _c.POINTER(_c.c_double)]
            lib.dsa_quantize_e4m3_append.restype = S
            lib.dsa_quantize_e4m3_append.argtypes = [_P, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int64, _P, _P,
                                                     _c.c_int32, _c.c_int64, _P, _P, _c.c_size_t, _P]
            lib.dsa_read_device_flags.restype = S
            lib.dsa_read_device_flags.argtypes = [_P, _c.POINTER(_c.c_uint32), _P]
            lib.dsa_status_string.restype = _c.c_char_p
            lib.dsa_status_string.argtypes = [S]
            lib.dsa_last_error.restype = _c.c_char_p
            lib.dsa_last_error.argtypes = []
            lib.dsa_launch_count.restype = _c.c_uint64
            lib.dsa_launch_count.argtypes = []
            lib.dsa_trace_enable.restype = S
            lib.dsa_trace_enable.argtypes = [_c.c_int32]
            lib.dsa_trace_read.restype = _c.c_int32
            lib.dsa_trace_read.argtypes = [_c.POINTER(_c.c_int32), _c.POINTER(_c.c_float), _c.c_int32,
                                           _c.POINTER(_c.c_int32)]
            lib.dsa_trace_disable.restype = None
            lib.dsa_trace_disable.argtypes = []
            _lib = lib
    return _lib


def status_string(s: int) -> str:
    return load_library().dsa_status_string(s).decode()


def _check(status: int):
    if status != 0:
        raise DsaError(status, load_library().dsa_last_error().decode())


def _ptr(t):
    return None if t is None else _c.c_void_p(t.data_ptr())


def _stream():
    return _c.c_void_p(torch.cuda.current_stream().cuda_stream)


# --- workspace ----------------------------------------------------------------------

_ws = {}


def workspace(nbytes: int = WS_MIN, device=None) -> torch.Tensor:
    """A zero-initialised uint8 workspace on `device` of at least `nbytes` (cached, grown)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    t = _ws.get(dev)
    if t is None or t.numel() < nbytes:
        if t is not None:
            torch.cuda.current_stream(dev).synchronize()
        t = torch.zeros(max(nbytes, WS_MIN), dtype=torch.uint8, device=dev)
        _ws[dev] = t
    return t


def release_workspace():
    _ws.clear()


# --- struct builders ----------------------------------------------------------------

def _stride(t, dim: int) -> int:
    """Stride of `dim` in elements, or 0 (the library's dense default) for a dimension of size
    1, whose stride torch leaves arbitrary."""
    return t.stride(dim) if t.shape[dim] > 1 else 0


def _row_pitch(t) -> int:
    """Row pitch of a [B,S,width] KV tensor: its row stride, or its width when S == 1."""
    return t.stride(1) if t.shape[1] > 1 else t.shape[2]


def indexer_struct(ix: dict) -> IndexerArgs:
    """The C struct of an indexer operand dict.  q [B,T,H_I,d_I] and k [B,S,d_I] may be
    strided views along their token / sequence axes (a token's codes stay contiguous); w and
    the scales are dense."""
    q, k, w = ix["q"], ix["k"], ix["w"]
    B, T, HI, DI = q.shape
    fp8 = q.dtype == torch.float8_e4m3fn
    for t in (q, k, w):
        assert t.is_cuda
    assert q.stride(3) == 1 and (HI == 1 or q.stride(2) == DI), "the codes of one token must be contiguous"
    assert k.stride(2) == 1 and (k.shape[1] == 1 or k.stride(1) == DI), "the keys of one sequence must be contiguous"
    assert w.is_contiguous()
    qs, ks = ix.get("q_scale"), ix.get("k_scale")
    for t in (qs, ks):
        assert t is None or t.is_contiguous()
    return IndexerArgs(B, T, k.shape[1], HI, DI, DSA_E4M3 if fp8 else DSA_BF16, q.data_ptr(),
                       qs.data_ptr() if (fp8 and qs is not None) else None, w.data_ptr(),
                       k.data_ptr(), ks.data_ptr() if (fp8 and ks is not None) else None,
                       int(ix.get("q_pos0", 0)), int(ix.get("diag", 0)), _stride(q, 0), _stride(q, 1),
                       _stride(k, 0))


def attn_struct(at: dict) -> AttnArgs:
    """The C struct of an attention operand dict.  q [B,T,H,d_qk] may be strided along its
    batch and token axes (a query's heads contiguous); k / v [B,S,*] along their batch axis and
    row pitch (k_ld / v_ld = the row stride)."""
    q, k = at["q"], at["k"]
    v = at.get("v")
    B, T, H, DQK = q.shape
    for t in (q, k) + ((v,) if v is not None else ()):
        assert t.is_cuda and t.dtype == torch.bfloat16 and t.stride(-1) == 1
    assert H == 1 or q.stride(2) == DQK, "the heads of one query must be contiguous"
    vv = k if v is None else v
    return AttnArgs(B, T, k.shape[1], H, DQK, int(at["d_v"]), float(at["scale"]), q.data_ptr(),
                    k.data_ptr(), _row_pitch(k), vv.data_ptr(), _row_pitch(vv), _stride(q, 0), _stride(q, 1),
                    _stride(k, 0), _stride(vv, 0))


# --- calls --------------------------------------------------------------------------

def workspace_size(ix: dict | None, k: int) -> int:
    if ix is None:
        return WS_MIN
    a = indexer_struct(ix)
    return int(load_library().dsa_workspace_size(_c.byref(a), k))


def indexer_scores(ix: dict, out: torch.Tensor | None = None) -> torch.Tensor:
    """Materialised indexer scores [B,T,S] fp32 (-inf where not visible)."""
    lib = load_library()
    a = indexer_struct(ix)
    if out is None:
        out = torch.empty((a.B, a.T, a.S), dtype=torch.float32, device=ix["q"].device)
    ws = workspace(WS_MIN, out.device)
    _check(lib.dsa_indexer_scores(_c.byref(a), _ptr(out), out.shape[-1], _ptr(ws), ws.numel(),
                                  _stream()))
    return out


def dsa_topk(k: int, *, ix: dict | None = None, scores: torch.Tensor | None = None,
             q_pos0: int = 0, diag: int = 0, idx: torch.Tensor | None = None,
             ws: torch.Tensor | None = None) -> torch.Tensor:
    """Top-k positions [B,T,k] int32 from indexer operands (fused path) or a score buffer."""
    lib = load_library()
    if ix is not None:
        a = indexer_struct(ix)
        src = TopkSrc(TOPK_FROM_INDEXER, None, 0, _c.pointer(a))
        B, T, S, q_pos0, diag = a.B, a.T, a.S, a.q_pos0, a.diag
        dev = ix["q"].device
        need = int(lib.dsa_workspace_size(_c.byref(a), k))
    else:
        assert scores is not None and scores.dtype == torch.float32 and scores.is_cuda
        sc = scores if scores.dim() == 3 else scores[None]
        B, T, S = sc.shape
        assert sc.stride(2) == 1 and sc.stride(0) == T * sc.stride(1)
        src = TopkSrc(TOPK_FROM_SCORES, sc.data_ptr(), sc.stride(1), None)
        dev = scores.device
        need = int(lib.dsa_topk_workspace_size(B, T, S, q_pos0, diag, k))
    if idx is None:
        idx = torch.empty((B, T, k), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(need, dev)
    _check(lib.dsa_topk(_c.byref(src), B, T, S, q_pos0, diag, k, _ptr(idx), _ptr(ws), ws.numel(),
                        _stream()))
    return idx


def dsa_sparse_attn(at: dict, idx: torch.Tensor, out: torch.Tensor | None = None,
                    lse: torch.Tensor | bool | None = True, ws: torch.Tensor | None = None):
    """(out [B,T,H,d_v] bf16, lse [B,T,H] fp32 or None).  `ws`: a workspace to use instead of
    the cached one (uint8, zero-filled once)."""
    lib = load_library()
    a = attn_struct(at)
    dev = at["q"].device
    assert idx.dtype == torch.int32 and idx.is_contiguous() and idx.shape[:2] == (a.B, a.T)
    if out is None:
        out = torch.empty((a.B, a.T, a.H, a.d_v), dtype=torch.bfloat16, device=dev)
    if lse is True:
        lse = torch.empty((a.B, a.T, a.H), dtype=torch.float32, device=dev)
    elif lse is False:
        lse = None
    if ws is None:
        ws = workspace(int(lib.dsa_attn_workspace_size(_c.byref(a), idx.shape[-1])), dev)
    _check(lib.dsa_sparse_attn(_c.byref(a), _ptr(idx), idx.shape[-1], _ptr(out), _ptr(lse),
                               _ptr(ws), ws.numel(), _stream()))
    return out, lse


def indexshare_draft_forward(ix: dict, at: dict, k: int, out: torch.Tensor | None = None,
                             lse: torch.Tensor | bool | None = True, idx: torch.Tensor | None = None):
    """Draft steps of a multi-token-prediction layer in one call: `ix` is the first step's
    indexer (T = 1 query per sequence, the layer's key cache), `at` holds the n steps' queries
    as q [B,n,H,d_qk] over the shared KV.  Returns (out [B,n,H,d_v] bf16, lse [B,n,H] fp32 or
    None, idx [B,1,k] int32: the first step's selection, read by every step)."""
    lib = load_library()
    a = attn_struct(at)
    x = indexer_struct(ix)
    dev = at["q"].device
    if idx is None:
        idx = torch.empty((a.B, 1, k), dtype=torch.int32, device=dev)
    assert idx.dtype == torch.int32 and idx.is_contiguous() and idx.numel() == a.B * k
    if out is None:
        out = torch.empty((a.B, a.T, a.H, a.d_v), dtype=torch.bfloat16, device=dev)
    if lse is True:
        lse = torch.empty((a.B, a.T, a.H), dtype=torch.float32, device=dev)
    elif lse is False:
        lse = None
    ws = workspace(int(lib.indexshare_draft_workspace_size(_c.byref(x), _c.byref(a), k)), dev)
    _check(lib.indexshare_draft_forward(_c.byref(x), _c.byref(a), k, _ptr(idx), _ptr(out), _ptr(lse), _ptr(ws),
                                        ws.numel(), _stream()))
    return out, lse, idx


def _group_structs(layers, schedule: str, k: int, outs, lses, idx_bufs, with_lse: bool):
    lib = load_library()
    n = len(layers)
    arr = (Layer * n)()
    at0 = layers[0]["at"]
    B, T = at0["q"].shape[:2]
    dev = at0["q"].device
    n_full = schedule.count("F")
    if idx_bufs is None:
        idx_bufs = [torch.empty((B, T, k), dtype=torch.int32, device=dev) for _ in range(n_full)]
    if outs is None:
        outs = []
        for l in layers:
            q = l["at"]["q"]
            outs.append(torch.empty(q.shape[:3] + (int(l["at"]["d_v"]),), dtype=torch.bfloat16, device=dev))
    if lses is None:
        lses = [torch.empty(l["at"]["q"].shape[:3], dtype=torch.float32, device=dev) if with_lse else None
                for l in layers]
    for i, l in enumerate(layers):
        if i < len(schedule) and schedule[i] == "F" and l.get("ix") is not None:
            arr[i].ix = indexer_struct(l["ix"])
        arr[i].at = attn_struct(l["at"])
        arr[i].out = outs[i].data_ptr()
        arr[i].lse = lses[i].data_ptr() if lses[i] is not None else None
    bufs = (_P * max(1, n_full))(*[b.data_ptr() for b in idx_bufs])
    need = int(lib.indexshare_group_workspace_size(arr, n, schedule.encode(), k, None)) if len(schedule) == n else WS_MIN
    return arr, bufs, need, outs, lses, idx_bufs, dev


def indexshare_group_forward(layers, schedule: str, k: int, outs=None, lses=None, idx_bufs=None,
                             with_lse: bool = True):
    """Run an F/S schedule over `layers` (dicts with 'ix' (F layers) and 'at').

    Returns (outs, lses, idx_bufs): per-layer outputs and LSEs, one idx buffer per F layer."""
    arr, bufs, need, outs, lses, idx_bufs, dev = _group_structs(layers, schedule, k, outs, lses, idx_bufs,
                                                                with_lse)
    ws = workspace(need, dev)
    _check(load_library().indexshare_group_forward(arr, len(layers), schedule.encode(), k, bufs, _ptr(ws),
                                                   ws.numel(), _stream()))
    return outs, lses, idx_bufs


def indexshare_group_forward_varlen(layers, schedule: str, k: int, cu_q, cu_k, q_pos0, outs=None, lses=None,
                                    idx_bufs=None, with_lse: bool = True):
    """indexshare_group_forward over sequences packed along the row axis: the layers' tensors
    are [1, total rows, ...] (queries, weights, outputs) and [1, total keys, ...] (keys, KV);
    sequence b owns query rows cu_q[b]:cu_q[b+1] and key rows cu_k[b]:cu_k[b+1], its first
    query at position q_pos0[b] (host integer sequences)."""
    lib = load_library()
    n_seqs = len(q_pos0)
    cq = (_c.c_int64 * (n_seqs + 1))(*[int(x) for x in cu_q])
    ck = (_c.c_int64 * (n_seqs + 1))(*[int(x) for x in cu_k])
    qp = (_c.c_int64 * n_seqs)(*[int(x) for x in q_pos0])
    seqs = Varlen(n_seqs, cq, ck, qp)
    arr, bufs, _, outs, lses, idx_bufs, dev = _group_structs(layers, schedule, k, outs, lses, idx_bufs, with_lse)
    need = int(lib.indexshare_group_workspace_size(arr, len(layers), schedule.encode(), k, _c.byref(seqs)))
    ws = workspace(need, dev)
    _check(lib.indexshare_group_forward_varlen(arr, len(layers), schedule.encode(), k, _c.byref(seqs), bufs,
                                               _ptr(ws), ws.numel(), _stream()))
    return outs, lses, idx_bufs


def topk_overlap(a: torch.Tensor, b: torch.Tensor, per_row: torch.Tensor | bool = True):
    """(per_row fp32 [rows] or None, mean) of |A and B| / |A| per row.  Synchronises."""
    lib = load_library()
    k = a.shape[-1]
    rows = a.numel() // k
    assert a.shape == b.shape and a.dtype == b.dtype == torch.int32
    a2, b2 = a.contiguous(), b.contiguous()
    if per_row is True:
        per_row = torch.empty(rows, dtype=torch.float32, device=a.device)
    elif per_row is False:
        per_row = None
    ws = workspace(WS_MIN + (0 if per_row is not None else rows * 4), a.device)
    mean = _c.c_double()
    _check(lib.topk_overlap(_ptr(a2), _ptr(b2), rows, k, _ptr(per_row), _c.byref(mean), _ptr(ws),
                            ws.numel(), _stream()))
    return per_row, mean.value


def topk_overlap_matrix(bufs, counts: bool = False):
    """All-pairs overlap of n index buffers of the same rows (the layer-overlap heatmap of an
    all-F pass): (M, counts) with M[i][j] = mean over rows of |A_i and A_j| / |A_i| as nested
    Python lists of floats, and counts an int32 [rows, n, n] device tensor of the per-row
    intersection sizes when asked for (else None).  Synchronises."""
    lib = load_library()
    n = len(bufs)
    k = bufs[0].shape[-1]
    rows = bufs[0].numel() // k
    for b in bufs:
        assert b.shape == bufs[0].shape and b.dtype == torch.int32 and b.is_contiguous()
    dev = bufs[0].device
    cnt = torch.empty((rows, n, n), dtype=torch.int32, device=dev) if counts else None
    arr = (_P * n)(*[b.data_ptr() for b in bufs])
    ws = workspace(int(lib.topk_overlap_matrix_workspace_size(n)), dev)
    out = (_c.c_double * (n * n))()
    _check(lib.topk_overlap_matrix(arr, n, rows, k, _ptr(cnt), out, _ptr(ws), ws.numel(), _stream()))
    return [[out[i * n + j] for j in range(n)] for i in range(n)], cnt


def _matrix_arg(M):
    n = len(M)
    flat = (_c.c_double * (n * n))(*[float(M[i][j]) for i in range(n) for j in range(n)])
    return n, flat


def indexshare_schedule_score(M, schedule: str) -> float:
    """Mean over layers of the overlap each layer keeps under `schedule` (host only)."""
    n, flat = _matrix_arg(M)
    v = _c.c_double()
    _check(load_library().indexshare_schedule_score(flat, n, schedule.encode(), _c.byref(v)))
    return v.value


def indexshare_schedule_search(M, n_full: int):
    """(schedule, score): a best schedule with n_full full layers under overlap matrix M."""
    n, flat = _matrix_arg(M)
    buf = _c.create_string_buffer(n + 1)
    v = _c.c_double()
    _check(load_library().indexshare_schedule_search(flat, n, int(n_full), buf, _c.byref(v)))
    return buf.value.decode(), v.value


def dsa_quantize_e4m3_append(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, pos0: int = 0,
                             positions: torch.Tensor | None = None):
    """Quantise x [B, n, width] bf16 to e4m3 with one fp32 scale per row and write the rows into
    codes [B, S_cap, width] (uint8 or float8_e4m3fn) / scales [B, S_cap] at row pos0 (or at
    positions[b], an int64 device tensor [B]) of every sequence."""
    assert x.dtype == torch.bfloat16 and x.dim() == 3 and x.stride(2) == 1 and x.stride(1) == x.shape[2]
    assert codes.dtype in (torch.uint8, torch.float8_e4m3fn) and codes.is_contiguous()
    assert scales.dtype == torch.float32 and scales.is_contiguous()
    B, n, width = x.shape
    assert codes.shape[0] == B and codes.shape[2] == width and scales.shape == codes.shape[:2]
    if positions is not None:
        assert positions.dtype == torch.int64 and positions.numel() == B and positions.is_contiguous()
    ws = workspace(WS_MIN, x.device)
    _check(load_library().dsa_quantize_e4m3_append(_ptr(x), B, n, width, x.stride(0), _ptr(codes), _ptr(scales),
                                                   codes.shape[1], int(pos0), _ptr(positions), _ptr(ws),
                                                   ws.numel(), _stream()))
    return codes, scales


def set_wait_limit(cycles: int) -> None:
    """Bound every wait inside the library's kernels launched from now on to `cycles` SM clock
    cycles (0: the default, about one second) -- dsa_set_wait_limit, for testing the timeout
    path."""
    load_library().dsa_set_wait_limit(int(cycles))


def topk_workspace_size(B: int, T: int, S: int, q_pos0: int, diag: int, k: int) -> int:
    """Workspace bytes dsa_topk over a score buffer uses for its fastest schedule."""
    return int(load_library().dsa_topk_workspace_size(B, T, S, q_pos0, diag, k))


def attn_workspace_size(at: dict, k: int) -> int:
    """Workspace bytes dsa_sparse_attn uses for its fastest schedule."""
    a = attn_struct(at)
    return int(load_library().dsa_attn_workspace_size(_c.byref(a), k))


def launch_count() -> int:
    """Kernels launched by the library since it was loaded."""
    return int(load_library().dsa_launch_count())


TRACE_KINDS = {1: "indexer", 2: "topk", 3: "attention", 4: "overlap"}


def trace_enable(max_launches: int = 4096) -> None:
    """Start bracketing every kernel launch with CUDA events (dsa_trace_enable)."""
    _check(load_library().dsa_trace_enable(int(max_launches)))


def trace_read(max_records: int = 1 << 16) -> list:
    """[(kind name, device ms), ...] of the launches recorded since the last read, in launch
    order; waits for them to finish.  Raises if the event pool dropped launches."""
    lib = load_library()
    kinds = (_c.c_int32 * max_records)()
    ms = (_c.c_float * max_records)()
    dropped = _c.c_int32(0)
    n = lib.dsa_trace_read(kinds, ms, max_records, _c.byref(dropped))
    if dropped.value:
        raise RuntimeError(f"dsa trace: {dropped.value} launches were not recorded (pool too small)")
    return [(TRACE_KINDS.get(kinds[i], str(kinds[i])), float(ms[i])) for i in range(n)]


def trace_disable() -> None:
    load_library().dsa_trace_disable()


def read_device_flags(device=None) -> int:
    """Flag word of the cached workspace (cleared by the read).  Synchronises."""
    lib = load_library()
    ws = workspace(WS_MIN, device)
    v = _c.c_uint32()
    _check(lib.dsa_read_device_flags(_ptr(ws), _c.byref(v), _stream()))
    return int(v.value)


__all__ = [
    "indexer_scores", "dsa_topk", "dsa_sparse_attn", "indexshare_group_forward", "topk_overlap",
    "topk_overlap_matrix", "indexshare_schedule_score", "indexshare_schedule_search",
    "dsa_quantize_e4m3_append", "indexshare_group_forward_varlen", "Varlen",
    "read_device_flags", "workspace", "workspace_size", "topk_workspace_size", "attn_workspace_size",
    "set_wait_limit", "load_library", "DsaError",
    "IndexerArgs", "AttnArgs", "TopkSrc", "Layer",
]
