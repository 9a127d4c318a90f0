"""Latent (MLA-style) cache on the GPU against the oracle.

latent_append must be byte-exact against ``oracle.mla.latent_append``, and
the decode call that appends each sequence's new latent itself must leave the
same pool and give the same result, bit for bit, as latent_append followed by
the decode call.  Decode over the latent pool (absorbed projections, attention over the
latents, up-projection) is compared with ``oracle.mla.mla_decode``, which
reconstructs every head's keys and values from the latents in fp64, at the
bf16 tolerance 2e-2."""
import pytest
import torch

import gpu_cases as G
from oracle import mla as M
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _workload(seed=11):
    return W.Workload("latent", torch.bfloat16, 1, 32, 1, 128, 16, 1, seed=seed, context=(1,))


def _run(w, lay, x, poison=False):
    pool = x.pool.clone()
    if poison:
        unused = ~G.used_slot_mask(lay, 16)
        pool[unused] = float("nan")
    slots = lay.slot_mapping[: lay.num_decode_tokens]
    gp = pool.cuda()
    B.latent_append(x.c_new.cuda(), gp, slots.cuda())
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    rp = G.cpu(pool).clone()
    M.latent_append(G.cpu(x.c_new), rp, slots)
    assert torch.equal(G.cpu(gp).view(torch.int16), rp.view(torch.int16))
    q = x.q.cuda()
    out = torch.empty_like(q)
    bt = lay.decode_block_table.cuda().contiguous()
    sl = lay.seq_lens.cuda()
    B.mla_decode_attention(out, q, x.w_k.cuda(), x.w_v.cuda(), gp, bt, sl,
                           int(lay.seq_lens.max()), w.scale)
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    return G.cpu(out), rp


def test_mla_balanced_walk_nan_in_unused_rows():
    """80 seeded lengths in [1, 2500] (with 1, 64, 65, 512, 513): more than 8
    stages of 64 tokens per CTA, so the kernel cuts the sequences into equal
    per-CTA shares at arbitrary stage boundaries and the merge takes a
    varying number of pieces per sequence; NaN in every unused pool row."""
    w = _workload(seed=12)
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(1, 2501, (80,), generator=g).tolist()
    lens[:5] = [1, 64, 65, 512, 513]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_latent(w, lay)
    got, rp = _run(w, lay, x, poison=True)
    ref = M.mla_decode(G.cpu(x.q), G.cpu(x.w_k), G.cpu(x.w_v), rp, lay.decode_block_table,
                       lay.seq_lens, w.scale)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= TOL


def test_mla_edge_lengths_nan_in_unused_rows():
    """Block (16), stage (64) and split (512) boundaries and one token; NaN
    in every pool row no sequence uses."""
    w = _workload()
    lens = [1, 2, 15, 16, 17, 33, 63, 64, 65, 511, 512, 513, 1024, 1025, 1600]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_latent(w, lay)
    got, rp = _run(w, lay, x, poison=True)
    ref = M.mla_decode(G.cpu(x.q), G.cpu(x.w_k), G.cpu(x.w_v), rp, lay.decode_block_table,
                       lay.seq_lens, w.scale)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= TOL


@pytest.mark.parametrize("name", ["llama8b_decode", "ragged_prefill"])
def test_mla_full_size_sampled_sequences(name):
    """The batch and lengths of a full-size workload; every head of 8
    sampled sequences (including the longest and the shortest)."""
    base = W.WORKLOADS[name]
    w = W.Workload("latent_" + name, torch.bfloat16, 1, 32, 1, 128, 16, base.num_seqs,
                   seed=base.seed, context=base.context, context_loguniform=base.context_loguniform)
    lay = W.make_layout(w, prefill=(0, 0))
    x = W.draw_latent(w, lay, device="cuda")
    got, rp = _run(w, lay, x)
    lens = lay.seq_lens
    g = torch.Generator().manual_seed(5)
    seqs = sorted({int(lens.argmax()), int(lens.argmin()),
                   *torch.randperm(w.num_seqs, generator=g)[:6].tolist()})
    ref = M.mla_decode(G.cpu(x.q), G.cpu(x.w_k), G.cpu(x.w_v), rp, lay.decode_block_table, lens,
                       w.scale, seqs=seqs)
    assert G.max_err(got[seqs], ref) <= TOL


def test_mla_rejects_unsupported_shape_and_small_workspace():
    w = _workload()
    lay = W.make_layout(w, seq_lens_after=[5, 700], prefill=(0, 0))
    x = W.draw_latent(w, lay, device="cuda")
    out = torch.empty_like(x.q)
    bt = lay.decode_block_table.cuda().contiguous()
    sl = lay.seq_lens.cuda()
    with pytest.raises(B.PagedKVError) as e:
        B.mla_decode_attention(out[:, :16], x.q[:, :16].contiguous(), x.w_k[:16], x.w_v[:16],
                               x.pool, bt, sl, 700, w.scale)
    assert e.value.status == 5          # 16 query heads: no kernel
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.PagedKVError) as e:
        B.mla_decode_attention(out, x.q, x.w_k, x.w_v, x.pool, bt, sl, 700, w.scale, small)
    assert e.value.status == 3          # workspace too small


@pytest.mark.parametrize("lens", [
    [1, 2, 15, 16, 17, 33, 63, 64, 65, 127, 128, 129, 511, 512, 513, 1024, 1025, 1600],
    "random80"])
def test_mla_append_in_call_equals_append_then_decode(lens):
    """pkv_mla_decode_attention_append == pkv_latent_append at the new
    tokens' slots + pkv_mla_decode_attention: pools and outputs bit for bit
    (NaN in every unused pool row), and the output within the tolerance of
    the oracle."""
    w = _workload(seed=13)
    if lens == "random80":
        g = torch.Generator().manual_seed(6)
        lens = torch.randint(1, 2501, (80,), generator=g).tolist()
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_latent(w, lay)
    sep, rp = _run(w, lay, x, poison=True)
    pool = x.pool.clone()
    pool[~G.used_slot_mask(lay, 16)] = float("nan")
    gp = pool.cuda()
    q = x.q.cuda()
    out = torch.empty_like(q)
    B.mla_decode_attention(out, q, x.w_k.cuda(), x.w_v.cuda(), gp, lay.decode_block_table.cuda().contiguous(),
                           lay.seq_lens.cuda(), int(lay.seq_lens.max()), w.scale,
                           c_new=x.c_new.cuda())
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    assert torch.equal(G.cpu(gp).view(torch.int16), rp.view(torch.int16))
    assert torch.equal(G.cpu(out).view(torch.int16), sep.view(torch.int16))
    ref = M.mla_decode(G.cpu(x.q), G.cpu(x.w_k), G.cpu(x.w_v), rp, lay.decode_block_table,
                       lay.seq_lens, w.scale)
    assert G.max_err(G.cpu(out), ref) <= TOL


def test_mla_append_in_call_bad_block_id_is_reported():
    """A block-table entry outside the pool at a sequence's last position:
    the append skips it, the decode reads a valid block instead, and the error
    word reports DEVERR_BLOCK_RANGE (2); no fault, the pool outside that row
    untouched."""
    w = _workload(seed=14)
    lay = W.make_layout(w, seq_lens_after=[40, 300], prefill=(0, 0))
    x = W.draw_latent(w, lay, device="cuda")
    bt = lay.decode_block_table.clone().contiguous()
    bt[1, (300 - 1) // 16] = lay.num_blocks + 7
    before = x.pool.clone()
    out = torch.empty_like(x.q)
    B.mla_decode_attention(out, x.q, x.w_k, x.w_v, x.pool, bt.cuda(), lay.seq_lens.cuda(), 300,
                           w.scale, c_new=x.c_new)
    assert B.get_device_error() & 2
    # sequence 0's new latent landed; nothing else changed
    slot0 = int(lay.slot_mapping[0])
    changed = (x.pool.view(torch.int16) != before.view(torch.int16)).any(dim=-1).nonzero()
    assert [tuple(t) for t in changed.tolist()] in ([], [(slot0 // 16, slot0 % 16)])
    assert torch.equal(x.pool[slot0 // 16, slot0 % 16].view(torch.int16),
                       x.c_new[0].view(torch.int16))
