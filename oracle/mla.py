"""Latent (MLA-style) KV cache for the oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` load it.

"The KV cache and prefix caching", section "What prefill stores and decode
reads", names multi-head latent attention (the DeepSeek line) as storing a
low-rank projection in place of the full keys and values.  The pages give no
rank and no formula; the reading used here:

  * per token and layer the cache holds one latent vector c of rank r;
  * query head h's key and value are up-projections of it,
    k_h = W_K[h] c and v_h = W_V[h] c, with W_K[h], W_V[h] of shape [D, r];
  * decode for head h is ordinary attention over every stored token:
    o_h = sum_j softmax_j(scale * q_h . k_{j,h}) v_{j,h}.

This module computes exactly that, in fp64: it gathers each sequence's
latents through its block table, reconstructs K and V per head and attends
with the maximum subtracted.  Pinned by ``tests/test_mla_oracle.py``.
"""
from __future__ import annotations

import torch


def latent_append(c_new: torch.Tensor, pool: torch.Tensor, slot_mapping: torch.Tensor) -> None:
    """Scatter c_new [T, r] into pool [NB, bs, r] in place (byte copy);
    slot = block * bs + row, negative slots are skipped."""
    bs = pool.shape[1]
    for t, slot in enumerate(slot_mapping.tolist()):
        if slot < 0:
            continue
        pool[slot // bs, slot % bs] = c_new[t]


def gather_latents(pool: torch.Tensor, block_table_row: torch.Tensor, n: int) -> torch.Tensor:
    """The first n latents of one sequence, [n, r] fp64, in position order."""
    bs = pool.shape[1]
    pos = torch.arange(n)
    blocks = block_table_row.to(torch.int64)[pos // bs]
    return pool[blocks, pos % bs].to(torch.float64)


def mla_decode(q, w_k, w_v, pool, block_table, seq_lens, scale, seqs=None) -> torch.Tensor:
    """q [B, Hq, D]; w_k, w_v [Hq, D, r]; pool [NB, bs, r]; block_table
    [B, max_blocks]; seq_lens [B] (tokens stored, after the append).
    Returns [len(seqs), Hq, D] float64 (all sequences by default)."""
    seqs = range(q.shape[0]) if seqs is None else seqs
    wk = w_k.to(torch.float64)
    wv = w_v.to(torch.float64)
    outs = []
    for b in seqs:
        n = int(seq_lens[b])
        c = gather_latents(pool, block_table[b], n)              # [n, r]
        qb = q[b].to(torch.float64)
        o = torch.empty(q.shape[1], q.shape[2], dtype=torch.float64)
        for h in range(q.shape[1]):
            k = c @ wk[h].T                                      # [n, D]: k_j = W_K[h] c_j
            v = c @ wv[h].T
            s = (k @ qb[h]) * scale
            p = torch.exp(s - s.max())
            o[h] = (p / p.sum()) @ v
        outs.append(o)
    return torch.stack(outs)


def latent_bytes_per_token(layers: int, rank: int, dtype_bytes: int = 2) -> int:
    """Cache bytes one token costs with a latent of the given rank."""
    return layers * rank * dtype_bytes
