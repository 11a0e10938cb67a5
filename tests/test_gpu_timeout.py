"""The bounded-wait path on the GPU, made to run out on purpose without touching the GPU's
state: with dsa_set_wait_limit(1) every wait that is not already complete gives up at once,
so each kernel stops its work, lets the copies and tensor-core products it has started
finish, frees its tensor memory and raises DSA_FLAG_TIMEOUT.  A normal call on the same
process afterwards must still match the oracle."""
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
    yield
    dsa.set_wait_limit(0)


def _run_all(ix, sc, at, idx, k):
    """The three kernels that wait on barriers: the indexer (TMA ring, MMA, epilogue), the
    top-k's bulk-copy ring (rows longer than 4,096 scores) and the tcgen05 attention."""
    a = dsa.dsa_topk(k, ix=ix)
    b = dsa.dsa_topk(k, scores=sc[None], q_pos0=sc.shape[1] - sc.shape[0])
    o, l = dsa.dsa_sparse_attn(at, idx)
    torch.cuda.synchronize()
    return a, b, o, l


def test_waits_that_run_out_raise_the_flag_and_leave_the_gpu_usable():
    wl = synth.WORKLOADS["prefill_16k"].replace(T=64, S=8192, q_pos0=8192 - 64, idx_dtype="e4m3",
                                                values="int", k=256)
    ix = synth.indexer_inputs(wl, 0, DEV)
    # 4,096 rows of 131,072 scores: every SM streams rows through rings of two copies, enough
    # traffic that some copy is still in flight when its consumer first looks
    sc = synth.scores_input(4096, 131072, DEV, "int", lo=-50, hi=50)
    at = synth.attn_inputs(wl.replace(T=160), 0, DEV)
    # the selecting path (scores never stored): 640 token blocks of rows longer than their
    # candidate room, so the indexer samples, sets thresholds and appends candidates
    wl_sel = wl.replace(T=2560, q_pos0=8192 - 2560)
    ix_sel = synth.indexer_inputs(wl_sel, 0, DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    idx = torch.sort(torch.randint(0, wl.S, (1, 160, wl.k), generator=g, device=DEV, dtype=torch.int32), -1).values
    try:
        dsa.set_wait_limit(1)
        _run_all(ix, sc, at, idx, wl.k)
        flags = dsa.read_device_flags()
    finally:
        dsa.set_wait_limit(0)
    assert flags & dsa.FLAG_TIMEOUT, hex(flags)
    # each kernel on its own raises the flag too
    for name, call in (("indexer + top-k", lambda: dsa.dsa_topk(wl.k, ix=ix)),
                       ("selecting indexer + top-k", lambda: dsa.dsa_topk(wl.k, ix=ix_sel)),
                       ("top-k over scores", lambda: dsa.dsa_topk(wl.k, scores=sc[None], q_pos0=131072 - 4096)),
                       ("attention", lambda: dsa.dsa_sparse_attn(at, idx))):
        raised = False
        for _ in range(3):  # a wait runs out only if its data is not there at the first look
            try:
                dsa.set_wait_limit(1)
                call()
                torch.cuda.synchronize()
            finally:
                dsa.set_wait_limit(0)
            flags = dsa.read_device_flags()  # read (and clear) after every attempt
            raised = raised or bool(flags & dsa.FLAG_TIMEOUT)
        assert raised, name
    # the same calls with the default bound: exact again, no flag
    a, b, o, l = _run_all(ix, sc, at, idx, wl.k)
    assert dsa.read_device_flags() == 0
    rows = [0, 13, 63]
    ref = oracle.indexer_topk(ix, wl.k, rows)
    assert np.array_equal(a.reshape(-1, wl.k)[rows].cpu().numpy(), ref)
    sel = dsa.dsa_topk(wl.k, ix=ix_sel)
    torch.cuda.synchronize()
    assert dsa.read_device_flags() == 0
    rows_sel = [0, 1283, 2559]
    ref_sel = oracle.indexer_topk(ix_sel, wl.k, rows_sel)
    assert np.array_equal(sel.reshape(-1, wl.k)[rows_sel].cpu().numpy(), ref_sel)
    some = [0, 1777, 4095]
    ref_b = oracle.topk_rows(sc[some].double().cpu().numpy(), np.array(some) + 131072 - 4096, wl.k)
    assert np.array_equal(b[0][some].cpu().numpy(), ref_b)
    host = dict(q_rows=at["q"].reshape(-1, wl.H, wl.DQK)[rows].cpu(), k=at["k"].cpu(), v=None, d_v=wl.DV,
                scale=wl.scale, T=160)
    ref_o, _ = oracle.sparse_attn(host, idx.reshape(-1, wl.k)[rows].cpu().numpy(), rows)
    assert np.abs(o.reshape(-1, wl.H, wl.DV)[rows].float().cpu().numpy() - ref_o).max() <= 2e-2
