"""The allocation-free indexer -> top-k entry point, dsa_topk_indexer_noalloc.

Some callers cannot allocate device memory at the moment they call the library: code that
runs inside an allocator or memory-pool callback (allocating there would re-enter the
allocator), plugins of runtimes that have already carved up all device memory, and
services that must keep a fixed footprint after start-up.  For them the library keeps the
scratch of this one path in a fixed 64 MiB device array of its own.  These tests call the
entry point through the C ABI (ctypes, device pointers from torch tensors) and check that
two calls in a row give exactly the index rows of dsa_topk(FROM_INDEXER), including a
shape that needs several passes through the fixed array, and that shapes too large for
the array are refused.  The file is collected last so that a failure here leaves every
other test already run.
"""
import ctypes

import pytest
import torch

import long_context_sparse_tcgen05_gb300 as dsa
from long_context_sparse_tcgen05_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
UNSUPPORTED = 2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_tcgen05_gb300 import build
    build.build()
    lib = dsa.load_library()
    lib.dsa_topk_indexer_noalloc.restype = ctypes.c_int
    lib.dsa_topk_indexer_noalloc.argtypes = [ctypes.POINTER(dsa.IndexerArgs), ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def _noalloc(lib, ix: dict, k: int, flags=None) -> torch.Tensor:
    a = dsa.indexer_struct(ix)
    idx = torch.full((a.B, a.T, k), -7, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dsa_topk_indexer_noalloc(ctypes.byref(a), k, ctypes.c_void_p(idx.data_ptr()),
                                      None if flags is None else ctypes.c_void_p(flags.data_ptr()), stream)
    assert st == 0, lib.dsa_last_error().decode()
    return idx


CASES = [
    # (workload, overrides, k): integer scores (ties everywhere), Gaussian bf16, and an FP8
    # prefix of a long sequence whose rows need three passes through the 64 MiB array
    ("tiny_l1k", dict(T=600, S=600), 64),
    ("prefill_16k", dict(T=700, S=700, values="gauss"), 256),
    ("prefill_128k", dict(T=300, S=131072, q_pos0=131072 - 300, values="gauss"), 2048),
]


@pytest.mark.parametrize("name,over,k", CASES)
def test_noalloc_matches_workspace_entry_point_twice(lib, name, over, k):
    wl = synth.WORKLOADS[name].replace(**over)
    ix = synth.indexer_inputs(wl, 0, DEV)
    ref = dsa.dsa_topk(k, ix=ix)
    first = _noalloc(lib, ix, k)
    second = _noalloc(lib, ix, k)
    torch.cuda.synchronize()
    assert torch.equal(first, ref)
    assert torch.equal(second, ref)


def test_noalloc_splits_few_long_rows_like_the_workspace_path(lib):
    """Decode shape (32 sequences x one query over 200,000 keys): the fixed array holds the
    25.6 MB of scores and, after them, the room of the few-long-rows top-k, so the call launches
    the indexer, the sampled threshold, the filter, the candidate top-k and the gated pass for
    rows the candidates could not finish -- and equals dsa_topk."""
    wl = synth.WORKLOADS["decode_b32_200k"].replace(values="gauss")
    ix = synth.indexer_inputs(wl, 0, DEV)
    ref = dsa.dsa_topk(wl.k, ix=ix)
    torch.cuda.synchronize()
    n0 = dsa.launch_count()
    got = _noalloc(lib, ix, wl.k)
    torch.cuda.synchronize()
    assert dsa.launch_count() - n0 == 5
    assert torch.equal(got, ref)
    del ix
    torch.cuda.empty_cache()


def test_noalloc_reports_flags_into_caller_word(lib):
    wl = synth.WORKLOADS["tiny_l1k"].replace(T=200, S=200)
    ix = synth.indexer_inputs(wl, 0, DEV)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = _noalloc(lib, ix, 32, flags)
    assert torch.equal(idx, dsa.dsa_topk(32, ix=ix))
    assert int(flags.item()) == 0


def test_noalloc_refuses_shapes_beyond_the_static_array(lib):
    wl = synth.WORKLOADS["tiny_l1k"].replace(T=4, S=64)
    ix = synth.indexer_inputs(wl, 0, DEV)
    a = dsa.indexer_struct(ix)
    a.B, a.S = 1, (64 << 20) // 4  # one score row alone would fill the whole array
    idx = torch.empty(4 * 16, dtype=torch.int32, device=DEV)
    st = lib.dsa_topk_indexer_noalloc(ctypes.byref(a), 16, ctypes.c_void_p(idx.data_ptr()), None, None)
    assert st == UNSUPPORTED
    assert "64 MiB" in lib.dsa_last_error().decode()
