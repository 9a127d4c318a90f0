"""Prefix caching end to end on the GPU: a second prompt that shares a system
prompt with a cached one reuses the cached blocks (found through the chained
block identifiers) and prefills only from the first unmatched block; its
output rows equal full causal attention over the whole logical sequence
("The KV cache and prefix caching": a server that has seen the prefix starts
prefill after it)."""
import random

import pytest
import torch

import gpu_cases as G
import oracle
from paged_kv_cache_104_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _tokens(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 128256) for _ in range(n)]


@pytest.mark.parametrize("dtype,hq,hkv,shared,len_b", [
    (torch.bfloat16, 8, 2, 1800, 2000), (torch.bfloat16, 4, 4, 200, 230),
    (torch.float32, 4, 2, 64, 65), (torch.bfloat16, 8, 2, 10, 300)])
def test_prefill_after_cached_prefix(dtype, hq, hkv, shared, len_b):
    d, bs = (128 if dtype == torch.bfloat16 else 16), 16
    w = G.custom_workload(dtype, hq, hkv, d, seed=61)
    system = _tokens(shared, 1)
    tok_a = system + _tokens(300, 2)
    tok_b = system + _tokens(len_b - shared, 3)
    g = torch.Generator().manual_seed(62)
    # logical K/V: a real model gives equal K/V for equal prefixes, so B's
    # first `shared` positions carry A's values
    k_a = torch.randn(len(tok_a), hkv, d, generator=g).to(dtype)
    v_a = torch.randn(len(tok_a), hkv, d, generator=g).to(dtype)
    k_b = torch.cat([k_a[:shared], torch.randn(len_b - shared, hkv, d, generator=g).to(dtype)])
    v_b = torch.cat([v_a[:shared], torch.randn(len_b - shared, hkv, d, generator=g).to(dtype)])
    q_b = torch.randn(len_b, hq, d, generator=g).to(dtype)

    nb_a = -(-len(tok_a) // bs)
    nb_b = -(-len_b // bs)
    num_blocks = nb_a + nb_b + 4
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    bt_a = perm[:nb_a]
    kc = torch.randn(num_blocks, hkv, bs, d, generator=g).to(dtype).cuda()
    vc = torch.randn(num_blocks, hkv, bs, d, generator=g).to(dtype).cuda()
    slots_a = torch.tensor([int(bt_a[p // bs]) * bs + p % bs for p in range(len(tok_a))])
    B.kv_append(k_a.cuda(), v_a.cuda(), kc, vc, slots_a.cuda())

    cache = B.PrefixCache()
    ids_a = B.prefix_hash_blocks(tok_a)
    cache.insert(ids_a, bt_a[:len(ids_a)].tolist())
    reused, blocks, _ = cache.plan(tok_b)
    assert reused == (min(shared, len_b - 1) // bs) * bs
    assert blocks == bt_a[:reused // bs].tolist()

    # B's table: the reused blocks, then fresh ones for everything after
    fresh = perm[nb_a:nb_a + nb_b - reused // bs]
    bt_b = torch.cat([torch.tensor(blocks, dtype=torch.int32), fresh])
    slots_b = torch.tensor([int(bt_b[p // bs]) * bs + p % bs for p in range(reused, len_b)])
    B.kv_append(k_b[reused:].cuda(), v_b[reused:].cuda(), kc, vc, slots_b.cuda())
    out = G.gpu_prefill(w, q_b[reused:], kc, vc, bt_b, reused)

    ref = oracle.causal_attention(q_b, k_b, v_b, w.scale)[reused:]
    assert G.max_err(out, ref) <= G.TOL[dtype]
    # the cached sequence's rows are unchanged: B's append wrote only fresh blocks
    kc_h = kc.cpu()
    for p in range(len(tok_a)):
        assert torch.equal(kc_h[int(bt_a[p // bs]), :, p % bs], k_a[p]), p
