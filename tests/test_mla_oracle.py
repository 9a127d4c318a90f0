"""The latent-cache oracle (``oracle/mla.py``) against facts fixed outside it
(CPU only).

  * identity up-projections turn it into grouped-query decode with one KV
    head whose key and value are both the latent -> the pinned GQA oracle;
  * one stored token returns W_V[h] c exactly (a softmax over one key is 1);
  * a pure-Python brute force with random projections (catches a transposed
    or swapped projection, a wrong scale or a wrong gather);
  * the append scatters rows exactly where block * 16 + row says.
"""
import math

import torch

import oracle
from oracle import mla as M
from paged_kv_cache_104_gb300 import workloads as W


def _layout(lens, hq=4, r=16, seed=0):
    w = W.Workload("mla_tiny", torch.float64, 1, hq, 1, r, 16, len(lens), seed=seed,
                   context=tuple(n - 1 for n in lens))
    return w, W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))


def _pool(lay, r, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(lay.num_blocks, 16, r, generator=g, dtype=torch.float64)


def test_identity_projections_reduce_to_gqa_decode():
    lens = [1, 17, 40, 77]
    hq, r = 4, 16
    w, lay = _layout(lens, hq, r)
    pool = _pool(lay, r, 1)
    g = torch.Generator().manual_seed(2)
    q = torch.randn(len(lens), hq, r, generator=g, dtype=torch.float64)
    eye = torch.eye(r, dtype=torch.float64).expand(hq, r, r).contiguous()
    got = M.mla_decode(q, eye, eye, pool, lay.block_table, lay.seq_lens, 1 / math.sqrt(r))
    kv = pool[:, None].contiguous()          # [NB, 1 KV head, 16, r]
    ref = oracle.paged_decode(q, kv, kv, lay.block_table, lay.seq_lens, 1 / math.sqrt(r))
    assert torch.allclose(got, ref, atol=1e-12, rtol=0)


def test_single_token_returns_projected_value():
    hq, d, r = 3, 8, 12
    w, lay = _layout([1, 1], hq, r)
    pool = _pool(lay, r, 3)
    g = torch.Generator().manual_seed(4)
    q = torch.randn(2, hq, d, generator=g, dtype=torch.float64)
    wk = torch.randn(hq, d, r, generator=g, dtype=torch.float64)
    wv = torch.randn(hq, d, r, generator=g, dtype=torch.float64)
    got = M.mla_decode(q, wk, wv, pool, lay.block_table, lay.seq_lens, 0.37)
    for b in range(2):
        c = pool[int(lay.block_table[b, 0]), 0]
        for h in range(hq):
            assert torch.allclose(got[b, h], wv[h] @ c, atol=1e-12, rtol=0)


def _brute(q, wk, wv, pool, bt, lens, scale):
    B, H, D = q.shape
    r = pool.shape[2]
    out = torch.zeros(B, H, D, dtype=torch.float64)
    for b in range(B):
        n = int(lens[b])
        cs = []
        for p in range(n):
            blk = int(bt[b, p // 16])
            cs.append([float(x) for x in pool[blk, p % 16]])
        for h in range(H):
            ks = [[sum(float(wk[h, d, i]) * c[i] for i in range(r)) for d in range(D)] for c in cs]
            vs = [[sum(float(wv[h, d, i]) * c[i] for i in range(r)) for d in range(D)] for c in cs]
            s = [scale * sum(float(q[b, h, d]) * k[d] for d in range(D)) for k in ks]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            z = sum(e)
            for d in range(D):
                out[b, h, d] = sum(e[j] * vs[j][d] for j in range(n)) / z
    return out


def test_brute_force_random_projections():
    lens = [3, 18]
    hq, d, r = 2, 5, 7
    w, lay = _layout(lens, hq, r, seed=5)
    pool = _pool(lay, r, 6)
    g = torch.Generator().manual_seed(7)
    q = torch.randn(2, hq, d, generator=g, dtype=torch.float64)
    wk = torch.randn(hq, d, r, generator=g, dtype=torch.float64)
    wv = torch.randn(hq, d, r, generator=g, dtype=torch.float64)
    got = M.mla_decode(q, wk, wv, pool, lay.block_table, lay.seq_lens, 0.41)
    ref = _brute(q, wk, wv, pool, lay.block_table, lay.seq_lens, 0.41)
    assert torch.allclose(got, ref, atol=1e-12, rtol=0)


def test_latent_append_against_indexing():
    lens = [5, 20]
    w, lay = _layout(lens, 2, 8)
    pool = torch.zeros(lay.num_blocks, 16, 8, dtype=torch.float32)
    c = torch.arange(2 * 8, dtype=torch.float32).reshape(2, 8) + 1
    slots = lay.slot_mapping.clone()
    M.latent_append(c, pool, slots)
    for t, s in enumerate(slots.tolist()):
        assert torch.equal(pool[s // 16, s % 16], c[t])
    assert int((pool != 0).sum()) == 16


def test_latent_bytes():
    # rank 128 in bf16 over 32 layers: 8 KiB per token, 1/16 of the
    # 131,072 bytes the GQA cache of the same model needs
    assert M.latent_bytes_per_token(32, 128) * 16 == oracle.kv_bytes_per_token(32, 8, 128)
