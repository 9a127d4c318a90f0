"""Chunked-prefill attention on the GPU against the fp64 oracle.

bf16 with head_dim 128 runs the tcgen05 kernel; fp32 runs the CUDA-core
kernel.  Tolerances as for decode (2e-2 bf16, 1e-5 fp32)."""
import pytest
import torch

import gpu_cases as G
import oracle
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _prefill_case(dtype, hq, hkv, d, prior, chunk, poison=True, seed=21, rows=None):
    w = G.custom_workload(dtype, hq, hkv, d, seed=seed)
    lay = W.make_layout(w, seq_lens_after=[1], prefill=(prior, chunk))
    x = W.draw_layer(w, lay, 0)
    if poison:
        G.poison_unused(x.k_cache, x.v_cache,
                        G.used_slot_mask(lay, w.block_size, prefill_len=prior + chunk))
    kc, vc = G.gpu_append(lay, x)
    rk, rv = G.oracle_append(lay, x)
    bt = lay.block_table[lay.prefill_row]
    out = G.gpu_prefill(w, x.q_prefill, kc, vc, bt, prior)
    ref = oracle.chunked_prefill(x.q_prefill, rk, rv, bt, prior, w.scale, rows=rows)
    got = G.cpu(out)
    if rows is not None:
        got = torch.stack([got[i, h] for i, h in rows])
    return got, ref


@pytest.mark.parametrize("prior,chunk", [
    (0, 128), (0, 1), (0, 16), (0, 200), (100, 300), (128, 256), (16, 17), (4096 - 1000, 700),
    (37, 513)])
def test_prefill_tcgen05_small_heads(prior, chunk):
    """Ragged chunk tails, priors off every tile boundary, a stale tail in the
    last block (NaN in unused rows) and a single-row chunk."""
    got, ref = _prefill_case(torch.bfloat16, 4, 1, 128, prior, chunk)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= 2e-2


@pytest.mark.parametrize("prior,chunk", [(0, 200), (100, 300), (37, 513), (0, 128)])
def test_prefill_tcgen05_query_tile_pairs(prior, chunk):
    """Group size 1 (no pair of heads shares a KV head): each CTA takes two
    consecutive query tiles of one head; an odd tile count leaves the last
    CTA's second tile past the chunk (chunk 200, 513 and 128)."""
    got, ref = _prefill_case(torch.bfloat16, 4, 4, 128, prior, chunk)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= 2e-2


def test_prefill_tcgen05_gqa_heads():
    got, ref = _prefill_case(torch.bfloat16, 16, 4, 128, 300, 260)
    assert G.max_err(got, ref) <= 2e-2


def test_prefill_full_size_chunk_sampled():
    """The 2,048-token chunk over 4,096 cached tokens, 32/8 heads: sampled rows
    including the tile edges 0, 15, 16, 127, 128 and the last row 2047."""
    w = W.WORKLOADS["ragged_prefill"]
    rows = W.sample_pairs(w.prefill_chunk, w.num_q_heads, 320, seed=4,
                          must=[0, 15, 16, 127, 128, 1023, 1024, 2047])
    got, ref = _prefill_case(torch.bfloat16, 32, 8, 128, 4096, 2048, poison=False, rows=rows)
    assert G.max_err(got, ref) <= 2e-2


@pytest.mark.parametrize("prior,chunk", [(0, 40), (21, 19), (5, 300)])
def test_prefill_cuda_core_fp32(prior, chunk):
    got, ref = _prefill_case(torch.float32, 4, 2, 16, prior, chunk)
    assert G.max_err(got, ref) <= 1e-5


def test_prefill_chunking_invariance_and_decode_agreement():
    """Two chunks of 384 == one chunk of 768 (each vs the oracle), and the last
    row equals the decode output at that position."""
    w = G.custom_workload(torch.bfloat16, 8, 2, 128, seed=33)
    prior, chunk = 200, 768
    lay = W.make_layout(w, seq_lens_after=[1], prefill=(prior, chunk))
    x = W.draw_layer(w, lay, 0)
    kc, vc = G.gpu_append(lay, x)
    bt = lay.block_table[lay.prefill_row]
    whole = G.gpu_prefill(w, x.q_prefill, kc, vc, bt, prior)
    a = G.gpu_prefill(w, x.q_prefill[:384], kc, vc, bt, prior)
    b = G.gpu_prefill(w, x.q_prefill[384:], kc, vc, bt, prior + 384)
    halves = torch.cat([a, b])
    rk, rv = G.oracle_append(lay, x)
    ref = oracle.chunked_prefill(x.q_prefill, rk, rv, bt, prior, w.scale)
    assert G.max_err(whole, ref) <= 2e-2
    assert G.max_err(halves, ref) <= 2e-2
    n = prior + chunk
    dec = G.gpu_decode(w, x.q_prefill[-1:], kc, vc, bt[None, :], torch.tensor([n], dtype=torch.int32))
    assert G.max_err(dec[0], G.cpu(whole[-1]).double()) <= 2e-2
