"""Paged decode attention on the GPU against the fp64 oracle.

Tolerances: max abs error 1e-5 for fp32 storage, 2e-2 for bf16 storage with
fp32 accumulation.  The pools the CUDA path reads were written by its own
kv_append; the oracle reads pools written by its own scatter (and the two are
checked bit-equal in test_gpu_append)."""
import pytest
import torch

import gpu_cases as G
import oracle
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode_case(name, pairs=None, gen="cpu", poison=False):
    w = W.WORKLOADS[name]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0, device=gen)
    if poison:
        G.poison_unused(x.k_cache, x.v_cache, G.used_slot_mask(lay, w.block_size))
    kc, vc = G.gpu_append(lay, x)
    rk, rv = G.oracle_append(lay, x)
    out = G.gpu_decode(w, x.q_decode, kc, vc, lay.decode_block_table, lay.seq_lens)
    ref = oracle.paged_decode(G.cpu(x.q_decode), rk, rv, lay.decode_block_table, lay.seq_lens,
                              w.scale, pairs=pairs)
    got = G.cpu(out)
    if pairs is not None:
        got = torch.stack([got[b, h] for b, h in pairs])
    return w, got, ref


@pytest.mark.parametrize("name", ["tiny_fp32", "toy_decode"])
def test_decode_small_configs_full(name):
    w, got, ref = _decode_case(name, poison=True)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= G.TOL[w.dtype]


@pytest.mark.parametrize("name", ["llama8b_decode", "long_context"])
def test_decode_full_size_layer_full_compare(name):
    """One layer at full size, every (sequence, head) compared."""
    w, got, ref = _decode_case(name, gen="cuda")
    assert G.max_err(got, ref) <= G.TOL[w.dtype]


def test_decode_ragged_full_size_sampled():
    w = W.WORKLOADS["ragged_prefill"]
    lay = W.make_layout(w)
    lens = lay.seq_lens
    must = [int(lens.argmax()), int(lens.argmin())]
    pairs = W.sample_pairs(w.num_seqs, w.num_q_heads, 384, seed=3, must=must)
    pairs += [(must[0], h) for h in range(w.num_q_heads)]
    pairs = sorted(set(pairs))
    w, got, ref = _decode_case("ragged_prefill", pairs=pairs, gen="cuda")
    assert G.max_err(got, ref) <= G.TOL[w.dtype]


@pytest.mark.parametrize("dtype,hq,hkv,d", [
    (torch.bfloat16, 32, 8, 128), (torch.bfloat16, 8, 8, 128), (torch.bfloat16, 16, 8, 128),
    (torch.bfloat16, 16, 2, 128), (torch.bfloat16, 16, 1, 128), (torch.float32, 8, 2, 128),
    (torch.float32, 4, 2, 16),
    (torch.float32, 8, 1, 16), (torch.float32, 4, 4, 16)])
def test_decode_edge_lengths_and_groups(dtype, hq, hkv, d):
    """Lengths at block (16) and split (512) boundaries, one token, every
    compiled group size; NaN in every pool row no sequence uses."""
    w = G.custom_workload(dtype, hq, hkv, d)
    lens = [1, 2, 15, 16, 17, 33, 511, 512, 513, 1024, 1025, 1600]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    G.poison_unused(x.k_cache, x.v_cache, G.used_slot_mask(lay, w.block_size))
    kc, vc = G.gpu_append(lay, x)
    rk, rv = G.oracle_append(lay, x)
    out = G.gpu_decode(w, x.q_decode, kc, vc, lay.decode_block_table, lay.seq_lens)
    ref = oracle.paged_decode(x.q_decode, rk, rv, lay.decode_block_table, lay.seq_lens, w.scale)
    assert torch.isfinite(G.cpu(out)).all()
    assert G.max_err(out, ref) <= G.TOL[dtype]


def test_decode_block_permutation_invariance():
    """Two physical shuffles of the same logical cache give bit-identical output."""
    w = G.custom_workload(torch.bfloat16, 32, 8, 128)
    lens = [700, 33, 1200]
    g = torch.Generator().manual_seed(5)
    ks = [torch.randn(n, 8, 128, generator=g).to(torch.bfloat16) for n in lens]
    vs = [torch.randn(n, 8, 128, generator=g).to(torch.bfloat16) for n in lens]
    q = torch.randn(len(lens), 32, 128, generator=g).to(torch.bfloat16)
    outs = []
    for seed_off in (0, 9):
        lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0), seed_offset=seed_off)
        kc = torch.zeros(lay.num_blocks, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        for b, n in enumerate(lens):
            slots = torch.tensor([int(lay.block_table[b, p // 16]) * 16 + p % 16 for p in range(n)])
            B.kv_append(ks[b].cuda(), vs[b].cuda(), kc, vc, slots.cuda())
        outs.append(G.gpu_decode(w, q, kc, vc, lay.decode_block_table, lay.seq_lens))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_decode_split_partials_match_single_split():
    """Split-K invariance: the 512-token split path (decode) and the
    single-split path (chunk mode of the CUDA-core kernel) agree."""
    w = G.custom_workload(torch.float32, 8, 2, 128)
    n = 1500
    lay = W.make_layout(w, seq_lens_after=[n], prefill=(0, 0))
    g = torch.Generator().manual_seed(8)
    k = torch.randn(n, 2, 128, generator=g)
    v = torch.randn(n, 2, 128, generator=g)
    q = torch.randn(1, 8, 128, generator=g)
    kc = torch.zeros(lay.num_blocks, 2, 16, 128, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([int(lay.block_table[0, p // 16]) * 16 + p % 16 for p in range(n)])
    B.kv_append(k.cuda(), v.cuda(), kc, vc, slots.cuda())
    dec = G.gpu_decode(w, q, kc, vc, lay.decode_block_table, lay.seq_lens)
    one = G.gpu_prefill(w, q, kc, vc, lay.block_table[0], prior=n - 1)   # one row at position n-1
    assert G.max_err(dec, G.cpu(one).double()) <= 1e-5


def test_decode_reports_bad_block_id_without_fault():
    w = G.custom_workload(torch.bfloat16, 32, 8, 128)
    lay = W.make_layout(w, seq_lens_after=[100, 40], prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    kc, vc = G.gpu_append(lay, x)
    bt = lay.decode_block_table.clone()
    bt[0, 2] = lay.num_blocks + 5
    G.gpu_decode(w, x.q_decode, kc, vc, bt, lay.seq_lens, check_err=False)
    assert B.get_device_error() == 2
    # the other sequence is still right
    rk, rv = G.oracle_append(lay, x)
    out = G.gpu_decode(w, x.q_decode, kc, vc, lay.decode_block_table, lay.seq_lens)
    ref = oracle.paged_decode(x.q_decode, rk, rv, lay.decode_block_table, lay.seq_lens, w.scale)
    assert G.max_err(out, ref) <= 2e-2


def test_decode_reports_length_beyond_bound():
    w = G.custom_workload(torch.bfloat16, 32, 8, 128)
    lay = W.make_layout(w, seq_lens_after=[100, 40], prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    kc, vc = G.gpu_append(lay, x)
    G.gpu_decode(w, x.q_decode, kc, vc, lay.decode_block_table, lay.seq_lens, max_seq_len=64,
                 check_err=False)
    assert B.get_device_error() == 3


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 1)])
def test_fused_append_decode_matches_append_then_decode(hq, hkv):
    """The fused call writes the same pool bytes as kv_append (bit-exact
    against the oracle's scatter) and returns bit-identical attention to
    kv_append followed by paged_decode_attention; within tolerance of the oracle."""
    w = G.custom_workload(torch.bfloat16, hq, hkv, 128, seed=71)
    lens = [1, 2, 16, 17, 33, 511, 512, 513, 1025, 1600]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    G.poison_unused(x.k_cache, x.v_cache, G.used_slot_mask(lay, w.block_size))
    bt = lay.decode_block_table.cuda().contiguous()
    sl = lay.seq_lens.cuda()
    msl = int(lay.seq_lens.max())
    ws = B.decode_workspace(len(lens), hq, 128, msl)
    # fused
    kc, vc = x.k_cache.cuda(), x.v_cache.cuda()
    out_f = torch.empty_like(x.q_decode).cuda()
    B.paged_decode_attention_append(out_f, x.q_decode.cuda(), x.k_new.cuda(), x.v_new.cuda(), kc, vc,
                                    bt, sl, msl, w.scale, ws)
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    # separate
    kc2, vc2 = G.gpu_append(lay, x)
    out_s = G.gpu_decode(w, x.q_decode, kc2, vc2, lay.decode_block_table, lay.seq_lens)
    rk, rv = G.oracle_append(lay, x)
    bits = lambda t: t.cpu().view(torch.int16)
    assert torch.equal(bits(kc), bits(rk)) and torch.equal(bits(vc), bits(rv))
    assert torch.equal(bits(out_f), bits(out_s))
    ref = oracle.paged_decode(x.q_decode, rk, rv, lay.decode_block_table, lay.seq_lens, w.scale)
    assert G.max_err(out_f, ref) <= 2e-2


def _balanced_lens(seed):
    """48 seeded lengths in [1, 3000], with 1, 64, 65, 512 and 513 among
    them: 48 x 8 KV heads x about 24 stages of 64 tokens is more than 8 per
    CTA of the whole GPU's grid, so the bf16 decode takes its balanced walk,
    which cuts streams at arbitrary 64-token boundaries."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, 3001, (48,), generator=g).tolist()
    lens[:5] = [1, 64, 65, 512, 513]
    return lens


@pytest.mark.parametrize("seed", [0, 1])
def test_decode_balanced_walk_vs_oracle(seed):
    """The balanced walk (fused append, then the merge of a variable number of
    pieces per stream): pools bit-exact against the oracle's scatter, every
    output within the bf16 tolerance of the fp64 oracle, NaN in unused rows."""
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=80 + seed)
    lens = _balanced_lens(seed)
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    G.poison_unused(x.k_cache, x.v_cache, G.used_slot_mask(lay, w.block_size))
    kc, vc = x.k_cache.cuda(), x.v_cache.cuda()
    bt = lay.decode_block_table.cuda().contiguous()
    msl = int(lay.seq_lens.max())
    ws = B.decode_workspace(len(lens), 32, 128, msl)
    out = torch.empty_like(x.q_decode).cuda()
    B.paged_decode_attention_append(out, x.q_decode.cuda(), x.k_new.cuda(), x.v_new.cuda(), kc, vc,
                                    bt, lay.seq_lens.cuda(), msl, w.scale, ws)
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    rk, rv = G.oracle_append(lay, x)
    bits = lambda t: t.cpu().view(torch.int16)
    assert torch.equal(bits(kc), bits(rk)) and torch.equal(bits(vc), bits(rv))
    ref = oracle.paged_decode(x.q_decode, rk, rv, lay.decode_block_table, lay.seq_lens, w.scale)
    assert G.max_err(out, ref) <= 2e-2
    # the unfused call takes the same walk: identical bits
    out2 = G.gpu_decode(w, x.q_decode, kc, vc, lay.decode_block_table, lay.seq_lens)
    assert torch.equal(bits(out), bits(out2))


def test_decode_balanced_walk_reports_bad_block_id():
    """A bad block id in one sequence of a balanced batch: the error word says
    so and every other sequence is still right."""
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=83)
    lens = _balanced_lens(3)
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    kc, vc = G.gpu_append(lay, x)
    bt = lay.decode_block_table.clone()
    bad = 7
    bt[bad, 1] = lay.num_blocks + 3
    out = G.gpu_decode(w, x.q_decode, kc, vc, bt, lay.seq_lens, check_err=False)
    assert B.get_device_error() == 2
    rk, rv = G.oracle_append(lay, x)
    ref = oracle.paged_decode(x.q_decode, rk, rv, lay.decode_block_table, lay.seq_lens, w.scale)
    keep = [i for i in range(len(lens)) if i != bad]
    assert G.max_err(out[keep], ref[keep]) <= 2e-2


def test_fused_append_decode_rejects_fp32():
    w = G.custom_workload(torch.float32, 4, 2, 16)
    lay = W.make_layout(w, seq_lens_after=[5], prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    kc, vc = x.k_cache.cuda(), x.v_cache.cuda()
    with pytest.raises(B.PagedKVError) as e:
        B.paged_decode_attention_append(torch.empty_like(x.q_decode).cuda(), x.q_decode.cuda(),
                                        x.k_new.cuda(), x.v_new.cuda(), kc, vc,
                                        lay.decode_block_table.cuda(), lay.seq_lens.cuda(), 5,
                                        w.scale)
    assert e.value.status == 5
