"""The benchmark's algorithmic work counts (the numerators of every roofline figure) against
closed forms worked out independently for the measured workloads (CPU only)."""
import importlib.util
import os
import sys

import pytest

from long_context_sparse_tcgen05_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_indexer_flops_closed_form(bench):
    # prefill of L keys with strictly-preceding visibility: L(L-1)/2 pairs, 2*64*128 flop each
    L = 131072
    assert bench.indexer_flops(synth.WORKLOADS["prefill_128k"]) == L * (L - 1) / 2 * 2 * 64 * 128
    # the last 4,096 rows of a 1M-key sequence: row i sees S - 4096 + i keys
    S, T = 1048576, 4096
    pairs = T * (S - T) + T * (T - 1) / 2
    assert bench.indexer_flops(synth.WORKLOADS["chunked_prefill_1m"]) == pairs * 2 * 64 * 128
    # decode: 32 queries over 200,000 keys each
    assert bench.indexer_flops(synth.WORKLOADS["decode_b32_200k"]) == 32 * 200000 * 2 * 64 * 128


def test_attention_bytes_closed_form(bench):
    wl = synth.WORKLOADS["prefill_128k"]
    L, k = 131072, 2048
    # gathered latent rows: min(k, t) for row t, 1,152 bytes each
    gathered = sum(min(k, t) for t in range(L)) * 576 * 2
    fixed = L * (64 * 576 * 2 + 64 * 512 * 2 + k * 4 + 64 * 4)
    assert bench.attn_bytes(wl) == gathered + fixed
    # about 3.26e11 bytes per layer, of which 3.07e11 gathered
    assert abs(bench.attn_bytes(wl) - 3.26e11) / 3.26e11 < 0.01
    assert abs(gathered - 3.07e11) / 3.07e11 < 0.01


def test_decode_indexer_bytes_and_its_bound(bench):
    wl = synth.WORKLOADS["decode_b32_200k"]
    keys = 32 * 200000 * (128 + 4)                 # e4m3 key cache + its scales
    queries = 32 * (64 * 128 + 64 * 4 + 4)         # e4m3 queries, head weights, scale
    scores = 32 * 200000 * 4                        # one fp32 score per visible pair
    assert bench.indexer_bytes(wl) == keys + queries + scores
    # about 120 flop per byte: far under the FP8 ridge (3,828 TFLOP/s over 6.7 TB/s ~ 570)
    assert 100 < bench.indexer_flops(wl) / bench.indexer_bytes(wl) < 140
    prefill = synth.WORKLOADS["prefill_128k"]
    assert bench.indexer_flops(prefill) / bench.indexer_bytes(prefill) > 570
    # prefill keeps candidates only: no score bytes in its count
    assert not bench.stores_scores(prefill) and bench.stores_scores(wl)
    assert bench.indexer_bytes(prefill) == 131072 * (128 + 4) + 131072 * (64 * 128 + 64 * 4 + 4)
