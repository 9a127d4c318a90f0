"""Checks that pin the oracle to facts fixed outside itself.

Each ``check_*`` takes the oracle module as its argument, so the same checks
run against the real oracle (``test_oracle_pins.py``) and against copies of
it with a planted mistake (``test_oracle_mutants.py``), where at least one
check must fail.

What pins what:
  * golden sizes printed on the pages -> kv_bytes_per_token
  * pure-Python brute force over the paged pool (tiny shapes) -> decode
  * cached decode == full causal recompute on the unpaged sequence
    ("KV cache and continuous batching: 1,000 people ask AI", section "What
    our lab measured": identical tokens on both paths) -> decode, gather, append
  * closed forms: one stored key returns its value; identical keys return the
    mean of the values; q = 0 returns the mean; constant V returns V; two keys
    give the logistic weight of scale * (score gap) -> softmax, scale, sign
  * GQA with repeated KV heads == MHA ("The KV cache and prefix caching":
    several query heads share one key/value head) -> head mapping
  * torch scaled_dot_product_attention in fp64 (a library routine, third
    opinion) -> decode and prefill
  * prefill with prior 0 == textbook causal attention; chunking invariance
    ("The KV cache is not your bottleneck", section "The fix that mattered")
  * physical block permutation and garbage in unused blocks change nothing
    ("The KV cache and prefix caching": fixed blocks with a block table)
"""
from __future__ import annotations

import json
import math
import os

import torch

from paged_kv_cache_104_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_sizes.json")


# ---------------------------------------------------------------- helpers
def _paged_from_contiguous(O, k_seq, v_seq, w, lay_seed=0, garbage=None):
    """Scatter per-sequence contiguous K/V (lists of [n, Hkv, D]) into a
    shuffled pool through the oracle's kv_append; returns (pools, layout)."""
    lens = [k.shape[0] for k in k_seq]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0), seed_offset=lay_seed)
    hkv, d, bs = w.num_kv_heads, w.head_dim, w.block_size
    fill = float("nan") if garbage == "nan" else 0.0
    kc = torch.full((lay.num_blocks, hkv, bs, d), fill, dtype=k_seq[0].dtype)
    vc = torch.full_like(kc, fill)
    if garbage == "randn":
        g = torch.Generator().manual_seed(77 + lay_seed)
        kc = torch.randn(kc.shape, generator=g).to(kc.dtype)
        vc = torch.randn(kc.shape, generator=g).to(kc.dtype)
    for b, n in enumerate(lens):
        slots = [int(lay.block_table[b, p // bs]) * bs + p % bs for p in range(n)]
        O.kv_append(k_seq[b], v_seq[b], kc, vc, torch.tensor(slots, dtype=torch.int64))
    return kc, vc, lay


def _small_workload(hq=4, hkv=2, d=16, bs=16, dtype=torch.float64):
    # the oracle reads fp32 or bf16 storage; tests use fp32 for exactness
    return W.Workload("pin", torch.float32, 1, hq, hkv, d, bs, 1, seed=5, context=(1,))


def _gen(seed):
    return torch.Generator().manual_seed(seed)


# ---------------------------------------------------------------- sizes
def check_kv_bytes_golden(O):
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        assert O.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"],
                                    c["dtype_bytes"]) == c["bytes_per_token"], c["source"]
    per_tok = O.kv_bytes_per_token(32, 8, 128)
    for t in g["totals"]:
        got = per_tok * t["tokens"] * t["requests"] / 2 ** t["unit_pow2"]
        if t.get("page_inconsistent"):
            # the printed total is not what its own expression gives; it is
            # the size of ``reconciling_tokens`` tokens instead
            assert round(got, t["printed_decimals"]) != t["value"]
            got = per_tok * t["reconciling_tokens"] * t["requests"] / 2 ** t["unit_pow2"]
        assert round(got, t["printed_decimals"]) == t["value"], t["source"]
    cap = g["capacity"]
    tokens = cap["free_gib"] * 2 ** 30 / per_tok
    assert abs(tokens - cap["approx_tokens"]) / cap["approx_tokens"] < 0.01
    assert abs(tokens / cap["tokens_per_request"] - cap["approx_requests"]) < 5


# ---------------------------------------------------------------- brute force
def _brute_decode(q, kc, vc, bt, seq_lens, scale):
    """Pure-Python loops over the paged pool (reads the pool directly)."""
    B, Hq, D = q.shape
    _, Hkv, bs, _ = kc.shape
    G = Hq // Hkv
    ql, kl, vl, btl = q.tolist(), kc.tolist(), vc.tolist(), bt.tolist()
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        n = int(seq_lens[b])
        for h in range(Hq):
            g = h // G
            scores = []
            for p in range(n):
                krow = kl[btl[b][p // bs]][g][p % bs]
                scores.append(scale * sum(ql[b][h][d] * krow[d] for d in range(D)))
            mx = max(scores)
            e = [math.exp(s - mx) for s in scores]
            z = sum(e)
            for d in range(D):
                out[b][h][d] = sum(e[p] * vl[btl[b][p // bs]][g][p % bs][d]
                                   for p in range(n)) / z
    return torch.tensor(out, dtype=torch.float64)


def check_decode_brute_force_tiny(O):
    w = W.WORKLOADS["tiny_fp32"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0)
    kc, vc = x.k_cache.clone(), x.v_cache.clone()
    O.kv_append(x.k_new, x.v_new, kc, vc, lay.slot_mapping)
    got = O.paged_decode(x.q_decode, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    ref = _brute_decode(x.q_decode, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    assert torch.allclose(got, ref, rtol=0, atol=1e-12), (got - ref).abs().max()


def check_append_against_indexing(O):
    """kv_append equals the plain index assignment pool[slot//bs, :, slot%bs] = row,
    leaves every other byte untouched and skips negative slots."""
    w = W.WORKLOADS["tiny_fp32"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0)
    slots = lay.slot_mapping.clone()
    slots[1] = -1
    kc, vc = x.k_cache.clone(), x.v_cache.clone()
    O.kv_append(x.k_new, x.v_new, kc, vc, slots)
    kr, vr = x.k_cache.clone(), x.v_cache.clone()
    bs = w.block_size
    for t, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        kr[s // bs, :, s % bs, :] = x.k_new[t]
        vr[s // bs, :, s % bs, :] = x.v_new[t]
    assert torch.equal(kc.view(torch.int32), kr.view(torch.int32))
    assert torch.equal(vc.view(torch.int32), vr.view(torch.int32))


# ---------------------------------------------------------------- recompute
def check_decode_equals_recompute(O):
    """Decode over the paged cache at the last position of each sequence ==
    the last row of full causal attention recomputed on the unpaged sequence."""
    w = _small_workload(hq=8, hkv=2, d=16)
    g = _gen(11)
    lens = [1, 15, 16, 17, 40]
    qs = [torch.randn(n, w.num_q_heads, w.head_dim, generator=g) for n in lens]
    ks = [torch.randn(n, w.num_kv_heads, w.head_dim, generator=g) for n in lens]
    vs = [torch.randn(n, w.num_kv_heads, w.head_dim, generator=g) for n in lens]
    kc, vc, lay = _paged_from_contiguous(O, ks, vs, w, garbage="randn")
    q_last = torch.stack([q[-1] for q in qs])
    got = O.paged_decode(q_last, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    for b, n in enumerate(lens):
        full = O.causal_attention(qs[b], ks[b], vs[b], w.scale)
        assert torch.allclose(got[b], full[-1], rtol=0, atol=1e-12), b


# ---------------------------------------------------------------- closed forms
def check_single_key_returns_value(O):
    w = _small_workload()
    g = _gen(12)
    k = [torch.randn(1, 2, 16, generator=g)]
    v = [torch.randn(1, 2, 16, generator=g)]
    kc, vc, lay = _paged_from_contiguous(O, k, v, w, garbage="randn")
    q = torch.randn(1, 4, 16, generator=g) * 10
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    for h in range(4):
        assert torch.equal(got[0, h], v[0][0, h // 2].double()), h


def check_identical_keys_give_mean(O):
    w = _small_workload()
    g = _gen(13)
    n = 37
    k1 = torch.randn(1, 2, 16, generator=g)
    k = [k1.expand(n, 2, 16).contiguous()]
    v = [torch.randn(n, 2, 16, generator=g)]
    kc, vc, lay = _paged_from_contiguous(O, k, v, w)
    q = torch.randn(1, 4, 16, generator=g)
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    mean = v[0].double().mean(0)  # [Hkv, D]
    for h in range(4):
        assert torch.allclose(got[0, h], mean[h // 2], rtol=0, atol=1e-12), h


def check_zero_query_gives_mean(O):
    w = _small_workload()
    g = _gen(14)
    n = 50
    k = [torch.randn(n, 2, 16, generator=g) * 5]
    v = [torch.randn(n, 2, 16, generator=g)]
    kc, vc, lay = _paged_from_contiguous(O, k, v, w)
    q = torch.zeros(1, 4, 16)
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    mean = v[0].double().mean(0)
    for h in range(4):
        assert torch.allclose(got[0, h], mean[h // 2], rtol=0, atol=1e-12), h


def check_constant_values(O):
    w = _small_workload()
    g = _gen(15)
    n = 33
    k = [torch.randn(n, 2, 16, generator=g)]
    c = torch.randn(2, 16, generator=g)
    v = [c.expand(n, 2, 16).contiguous()]
    kc, vc, lay = _paged_from_contiguous(O, k, v, w)
    q = torch.randn(1, 4, 16, generator=g)
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    for h in range(4):
        assert torch.allclose(got[0, h], c[h // 2].double(), rtol=0, atol=1e-12), h


def check_two_key_logistic(O):
    """keys a*e0 and 0, query e0: weight of the first value is
    1 / (1 + exp(-scale * a)); fixes the scale and the sign."""
    w = _small_workload()
    a = 3.0
    k = torch.zeros(2, 2, 16)
    k[0, :, 0] = a
    v = torch.zeros(2, 2, 16)
    v[0, :, 1] = 1.0
    v[1, :, 2] = 1.0
    kc, vc, lay = _paged_from_contiguous(O, [k], [v], w)
    q = torch.zeros(1, 4, 16)
    q[0, :, 0] = 1.0
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    p1 = 1.0 / (1.0 + math.exp(-w.scale * a))
    for h in range(4):
        assert abs(float(got[0, h, 1]) - p1) < 1e-13
        assert abs(float(got[0, h, 2]) - (1 - p1)) < 1e-13


def check_gqa_equals_mha_with_repeated_heads(O):
    """GQA read as contiguous groups: query head h uses KV head h // G.
    Repeating each KV head G times and running MHA must give the same."""
    hq, hkv, d = 8, 2, 16
    G = hq // hkv
    w_g = _small_workload(hq, hkv, d)
    w_m = _small_workload(hq, hq, d)
    g = _gen(16)
    lens = [9, 30]
    ks = [torch.randn(n, hkv, d, generator=g) for n in lens]
    vs = [torch.randn(n, hkv, d, generator=g) for n in lens]
    q = torch.randn(len(lens), hq, d, generator=g)
    kc, vc, lay = _paged_from_contiguous(O, ks, vs, w_g)
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w_g.scale)
    km = [k.repeat_interleave(G, dim=1) for k in ks]
    vm = [v.repeat_interleave(G, dim=1) for v in vs]
    kc2, vc2, lay2 = _paged_from_contiguous(O, km, vm, w_m, lay_seed=3)
    ref = O.paged_decode(q, kc2, vc2, lay2.block_table, lay2.seq_lens, w_m.scale)
    assert torch.allclose(got, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- library
def _sdpa_causal(q, k, v, scale, G, prior=0):
    """torch SDPA in fp64 with the KV heads repeated; query row i sits at
    position prior + i over keys 0..prior+i."""
    qd = q.double().transpose(0, 1)                     # [Hq, C, D]
    kd = k.double().repeat_interleave(G, dim=1).transpose(0, 1)
    vd = v.double().repeat_interleave(G, dim=1).transpose(0, 1)
    C, T = q.shape[0], k.shape[0]
    mask = torch.arange(T)[None, :] <= (prior + torch.arange(C))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=scale)
    return o.transpose(0, 1)


def check_decode_against_sdpa(O):
    w = _small_workload(hq=8, hkv=4, d=32)
    g = _gen(17)
    lens = [3, 16, 31, 64]
    ks = [torch.randn(n, 4, 32, generator=g) for n in lens]
    vs = [torch.randn(n, 4, 32, generator=g) for n in lens]
    q = torch.randn(len(lens), 8, 32, generator=g)
    kc, vc, lay = _paged_from_contiguous(O, ks, vs, w, garbage="randn")
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    for b, n in enumerate(lens):
        ref = _sdpa_causal(q[b:b + 1], ks[b], vs[b], w.scale, 2, prior=n - 1)[0]
        assert torch.allclose(got[b], ref, rtol=0, atol=1e-12), b


def check_prefill_against_sdpa(O):
    w = _small_workload(hq=4, hkv=2, d=16)
    g = _gen(18)
    prior, chunk = 21, 19
    n = prior + chunk
    k = torch.randn(n, 2, 16, generator=g)
    v = torch.randn(n, 2, 16, generator=g)
    q = torch.randn(chunk, 4, 16, generator=g)
    kc, vc, lay = _paged_from_contiguous(O, [k], [v], w, garbage="randn")
    got = O.chunked_prefill(q, kc, vc, lay.block_table[0], prior, w.scale)
    ref = _sdpa_causal(q, k, v, w.scale, 2, prior=prior)
    assert torch.allclose(got, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- prefill
def check_prefill_prior0_is_causal_attention(O):
    w = _small_workload(hq=4, hkv=1, d=16)
    g = _gen(19)
    n = 45
    q = torch.randn(n, 4, 16, generator=g)
    k = torch.randn(n, 1, 16, generator=g)
    v = torch.randn(n, 1, 16, generator=g)
    kc, vc, lay = _paged_from_contiguous(O, [k], [v], w)
    got = O.chunked_prefill(q, kc, vc, lay.block_table[0], 0, w.scale)
    ref = O.causal_attention(q, k, v, w.scale)
    assert torch.allclose(got, ref, rtol=0, atol=1e-12)


def check_prefill_chunking_invariance(O):
    """Prefill in chunks of 7 (each over the cache the earlier chunks left) ==
    one chunk; and the last row == the decode output at that position."""
    w = _small_workload(hq=4, hkv=2, d=16)
    g = _gen(20)
    n = 37
    q = torch.randn(n, 4, 16, generator=g)
    k = torch.randn(n, 2, 16, generator=g)
    v = torch.randn(n, 2, 16, generator=g)
    kc, vc, lay = _paged_from_contiguous(O, [k], [v], w)
    bt = lay.block_table[0]
    whole = O.chunked_prefill(q, kc, vc, bt, 0, w.scale)
    parts = [O.chunked_prefill(q[s:s + 7], kc, vc, bt, s, w.scale) for s in range(0, n, 7)]
    assert torch.allclose(torch.cat(parts), whole, rtol=0, atol=1e-12)
    dec = O.paged_decode(q[-1:], kc, vc, lay.block_table[:1], torch.tensor([n]), w.scale)
    assert torch.allclose(dec[0], whole[-1], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- paging
def check_block_permutation_invariance(O):
    """Same logical sequences, two different shuffles of the physical pool
    (and NaN in every unused slot): identical results."""
    w = _small_workload(hq=4, hkv=2, d=16)
    g = _gen(21)
    lens = [5, 16, 17, 48]
    ks = [torch.randn(n, 2, 16, generator=g) for n in lens]
    vs = [torch.randn(n, 2, 16, generator=g) for n in lens]
    q = torch.randn(len(lens), 4, 16, generator=g)
    kc1, vc1, lay1 = _paged_from_contiguous(O, ks, vs, w, lay_seed=1, garbage="randn")
    kc2, vc2, lay2 = _paged_from_contiguous(O, ks, vs, w, lay_seed=2, garbage="nan")
    assert not torch.equal(lay1.block_table, lay2.block_table)
    o1 = O.paged_decode(q, kc1, vc1, lay1.block_table, lay1.seq_lens, w.scale)
    o2 = O.paged_decode(q, kc2, vc2, lay2.block_table, lay2.seq_lens, w.scale)
    assert torch.isfinite(o2).all()
    assert torch.equal(o1, o2)


def check_sampled_pairs_match_full(O):
    w = W.WORKLOADS["tiny_fp32"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0)
    kc, vc = x.k_cache.clone(), x.v_cache.clone()
    O.kv_append(x.k_new, x.v_new, kc, vc, lay.slot_mapping)
    full = O.paged_decode(x.q_decode, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    pairs = [(3, 1), (0, 2), (2, 3)]
    part = O.paged_decode(x.q_decode, kc, vc, lay.block_table, lay.seq_lens, w.scale, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert torch.equal(part[i], full[b, h])


def check_bf16_storage_widening(O):
    """bf16 storage is read exactly: bf16 inputs give the fp32 answer of the
    same (exactly representable) values."""
    w = _small_workload()
    g = _gen(22)
    k = [torch.randn(20, 2, 16, generator=g).to(torch.bfloat16)]
    v = [torch.randn(20, 2, 16, generator=g).to(torch.bfloat16)]
    q = torch.randn(1, 4, 16, generator=g).to(torch.bfloat16)
    kc, vc, lay = _paged_from_contiguous(O, k, v, w)
    got = O.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    kc32, vc32, lay32 = _paged_from_contiguous(O, [k[0].float()], [v[0].float()], w)
    ref = O.paged_decode(q.float(), kc32, vc32, lay32.block_table, lay32.seq_lens, w.scale)
    assert torch.equal(got, ref)


ALL_CHECKS = [
    check_kv_bytes_golden,
    check_decode_brute_force_tiny,
    check_append_against_indexing,
    check_decode_equals_recompute,
    check_single_key_returns_value,
    check_identical_keys_give_mean,
    check_zero_query_gives_mean,
    check_constant_values,
    check_two_key_logistic,
    check_gqa_equals_mha_with_repeated_heads,
    check_decode_against_sdpa,
    check_prefill_against_sdpa,
    check_prefill_prior0_is_causal_attention,
    check_prefill_chunking_invariance,
    check_block_permutation_invariance,
    check_sampled_pairs_match_full,
    check_bf16_storage_widening,
]
