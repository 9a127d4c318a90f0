"""One layer's decode and a prompt chunk's prefill run side by side on
disjoint SMs (pkv_decode_prefill_attention): the prefill as persistent CTAs on
prefill_sms SMs, the decode (with its fused append) on the rest.  The results
must equal those of the two calls made one after the other (kv_append of the
chunk, paged_decode_attention_append, chunked_prefill): the prefill and the
pools bit for bit, the decode bit for bit while both walk 512-token splits and
to rounding once the batch is large enough for the balanced walk the decode
takes when it runs alone; and stay within the bf16 tolerance of the oracle.
Given the chunk's new keys and values, the call appends them itself (the
append launched first, the prefill as its programmatic dependent): the same
results, bit for bit, as kv_append followed by the call."""
import pytest
import torch

import gpu_cases as G
import oracle
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().view(torch.int16)


def _run_both(w, lay, x, prior, prefill_sms, dev="cuda", chunk_in_call=False):
    """Serial calls, then the side-by-side call on a second copy of the pools
    (chunk_in_call: the call appends the chunk's keys and values itself);
    returns (serial decode, serial prefill, side decode, side prefill, pools)."""
    nd = lay.num_decode_tokens
    bt = lay.decode_block_table.to(dev).contiguous()
    sl = lay.seq_lens.to(dev)
    msl = int(lay.seq_lens.max())
    bt_pre = lay.block_table[lay.prefill_row].to(dev).contiguous()
    q_dec, q_pre = x.q_decode.to(dev), x.q_prefill.to(dev)
    k_dec, v_dec = x.k_new[:nd].to(dev), x.v_new[:nd].to(dev)
    k_pre, v_pre = x.k_new[nd:].to(dev), x.v_new[nd:].to(dev)
    slot_pre = lay.slot_mapping[nd:].to(dev)
    ws = B.decode_workspace(nd, w.num_q_heads, w.head_dim, msl, device=dev)
    outs = []
    pools = []
    for side in (False, True):
        kc, vc = x.k_cache.to(dev), x.v_cache.to(dev)
        if not (side and chunk_in_call):
            B.kv_append(k_pre, v_pre, kc, vc, slot_pre)
        od, op = torch.empty_like(q_dec), torch.empty_like(q_pre)
        if side and chunk_in_call:
            B.decode_prefill_attention(od, q_dec, k_dec, v_dec, kc, vc, bt, sl, msl, op, q_pre, bt_pre,
                                       prior, w.scale, ws, prefill_sms=prefill_sms,
                                       chunk_k_new=k_pre, chunk_v_new=v_pre, chunk_slots=slot_pre)
        elif side:
            B.decode_prefill_attention(od, q_dec, k_dec, v_dec, kc, vc, bt, sl, msl, op, q_pre, bt_pre,
                                       prior, w.scale, ws, prefill_sms=prefill_sms)
        else:
            B.paged_decode_attention_append(od, q_dec, k_dec, v_dec, kc, vc, bt, sl, msl, w.scale, ws)
            B.chunked_prefill_attention(op, q_pre, kc, vc, bt_pre, prior, w.scale)
        torch.cuda.synchronize()
        assert B.get_device_error() == 0
        outs += [od, op]
        pools.append((kc, vc))
    return outs, pools


@pytest.mark.parametrize("chunk_in_call", [False, True])
@pytest.mark.parametrize("prefill_sms", [8, 40, 100])
def test_side_by_side_equals_serial_and_oracle(prefill_sms, chunk_in_call):
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=91)
    lens = [1, 17, 300, 512, 513, 1500, 2600, 4097]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(700, 600))
    x = W.draw_layer(w, lay, 0)
    (sd, sp, bd, bp), pools = _run_both(w, lay, x, 700, prefill_sms, chunk_in_call=chunk_in_call)
    assert torch.equal(_bits(sd), _bits(bd)), "decode differs from the serial calls"
    assert torch.equal(_bits(sp), _bits(bp)), "prefill differs from the serial calls"
    (k1, v1), (k2, v2) = pools
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    rk, rv = G.oracle_append(lay, x)
    ref_d = oracle.paged_decode(x.q_decode, rk, rv, lay.decode_block_table, lay.seq_lens, w.scale)
    ref_p = oracle.chunked_prefill(x.q_prefill, rk, rv, lay.block_table[lay.prefill_row], 700,
                                   w.scale)
    assert G.max_err(bd, ref_d) <= 2e-2
    assert G.max_err(bp, ref_p) <= 2e-2


def test_side_by_side_full_size_layer():
    """The ragged 128-sequence batch with its 2,048-token chunk over 4,096
    cached tokens, 40 SMs for the prefill, the chunk appended by the call (as
    the bench's step runs it): the prefill and the pools equal to the serial
    calls bit for bit; the decode (512-token splits beside the prefill, the
    balanced walk alone) to within a bf16 rounding step of its values
    (|o| < 1)."""
    w = W.WORKLOADS["ragged_prefill"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0)
    (sd, sp, bd, bp), pools = _run_both(w, lay, x, w.prefill_prior, 40, chunk_in_call=True)
    assert torch.equal(_bits(sp), _bits(bp))
    (k1, v1), (k2, v2) = pools
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    assert float(sd.float().abs().max()) < 1.0
    assert G.max_err(bd, sd.cpu()) <= 2.0 ** -8


@pytest.mark.parametrize("hq,hkv", [(8, 8), (4, 4)])
def test_side_by_side_group_of_one(hq, hkv):
    """A GQA group of 1: the prefill pairs query tiles of one head instead of
    heads; still equal to the serial calls."""
    w = G.custom_workload(torch.bfloat16, hq, hkv, 128, seed=92)
    lay = W.make_layout(w, seq_lens_after=[5, 700, 1300], prefill=(130, 250))
    x = W.draw_layer(w, lay, 0)
    (sd, sp, bd, bp), _ = _run_both(w, lay, x, 130, 16)
    assert torch.equal(_bits(sd), _bits(bd)) and torch.equal(_bits(sp), _bits(bp))


def test_side_by_side_per_head_stages():
    """Two KV heads, too few for a group of four: beside the prefill the
    decode keeps one head per stage and 512-token splits; still equal to the
    serial calls."""
    w = G.custom_workload(torch.bfloat16, 16, 2, 128, seed=95)
    lay = W.make_layout(w, seq_lens_after=[5, 700, 1300], prefill=(130, 250))
    x = W.draw_layer(w, lay, 0)
    (sd, sp, bd, bp), _ = _run_both(w, lay, x, 130, 16)
    assert torch.equal(_bits(sd), _bits(bd)) and torch.equal(_bits(sp), _bits(bp))


def test_side_by_side_too_many_work_items_runs_serial():
    """514 work items (257 query tiles x 2 head pairs) exceed the persistent
    list: serial, same results."""
    w = G.custom_workload(torch.bfloat16, 4, 2, 128, seed=94)
    lay = W.make_layout(w, seq_lens_after=[9, 2000], prefill=(0, 257 * 128))
    x = W.draw_layer(w, lay, 0)
    for chunk_in_call in (False, True):
        (sd, sp, bd, bp), (p1, p2) = _run_both(w, lay, x, 0, 20, chunk_in_call=chunk_in_call)
        assert torch.equal(_bits(sd), _bits(bd)) and torch.equal(_bits(sp), _bits(bp))
        assert torch.equal(_bits(p1[0]), _bits(p2[0])) and torch.equal(_bits(p1[1]), _bits(p2[1]))


def test_side_by_side_prefill_sms_at_or_above_the_gpu():
    """prefill_sms at the SM count leaves nothing for the decode: serial."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = G.custom_workload(torch.bfloat16, 8, 2, 128, seed=93)
    lay = W.make_layout(w, seq_lens_after=[40, 900], prefill=(0, 300))
    x = W.draw_layer(w, lay, 0)
    for chunk_in_call in (False, True):
        (sd, sp, bd, bp), (p1, p2) = _run_both(w, lay, x, 0, sms, chunk_in_call=chunk_in_call)
        assert torch.equal(_bits(sd), _bits(bd)) and torch.equal(_bits(sp), _bits(bp))
        assert torch.equal(_bits(p1[0]), _bits(p2[0])) and torch.equal(_bits(p1[1]), _bits(p2[1]))


def test_side_by_side_rejects_fp32_and_bad_split():
    w = G.custom_workload(torch.float32, 4, 2, 128)
    lay = W.make_layout(w, seq_lens_after=[3], prefill=(0, 20))
    x = W.draw_layer(w, lay, 0)
    kc, vc = x.k_cache.cuda(), x.v_cache.cuda()
    bt = lay.decode_block_table.cuda().contiguous()
    ws = B.decode_workspace(1, 4, 128, 3)
    with pytest.raises(B.PagedKVError):
        B.decode_prefill_attention(torch.empty_like(x.q_decode).cuda(), x.q_decode.cuda(),
                                   x.k_new[:1].cuda(), x.v_new[:1].cuda(), kc, vc, bt,
                                   lay.seq_lens.cuda(), 3, torch.empty_like(x.q_prefill).cuda(),
                                   x.q_prefill.cuda(), lay.block_table[lay.prefill_row].cuda(), 0,
                                   w.scale, ws, prefill_sms=8)
    w = G.custom_workload(torch.bfloat16, 4, 2, 128)
    lay = W.make_layout(w, seq_lens_after=[3], prefill=(0, 20))
    x = W.draw_layer(w, lay, 0)
    with pytest.raises(B.PagedKVError):
        _run_both(w, lay, x, 0, -1)


def test_side_by_side_chunk_append_needs_all_three():
    """chunk_k_new, chunk_v_new and chunk_slots come together or not at all."""
    w = G.custom_workload(torch.bfloat16, 4, 2, 128)
    lay = W.make_layout(w, seq_lens_after=[30], prefill=(0, 20))
    x = W.draw_layer(w, lay, 0, device="cuda")
    nd = lay.num_decode_tokens
    bt = lay.decode_block_table.cuda().contiguous()
    ws = B.decode_workspace(1, 4, 128, 30)
    with pytest.raises(B.PagedKVError):
        B.decode_prefill_attention(torch.empty_like(x.q_decode), x.q_decode, x.k_new[:nd],
                                   x.v_new[:nd], x.k_cache, x.v_cache, bt, lay.seq_lens.cuda(), 30,
                                   torch.empty_like(x.q_prefill), x.q_prefill,
                                   lay.block_table[lay.prefill_row].cuda(), 0, w.scale, ws,
                                   prefill_sms=8, chunk_k_new=x.k_new[nd:])


def test_side_by_side_span_record():
    """pkv_set_span_buffer: the side-by-side call records each half's
    earliest CTA start and latest CTA end (ordered, the decode starting after
    the prefill it depends on), with the results unchanged bit for bit; None
    turns the record off again."""
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=95)
    lay = W.make_layout(w, seq_lens_after=[40, 900, 3000], prefill=(300, 400))
    x = W.draw_layer(w, lay, 0)
    (sd, sp, bd, bp), _ = _run_both(w, lay, x, 300, 40, chunk_in_call=True)
    span = torch.tensor([-1, 0, -1, 0], dtype=torch.int64, device="cuda")
    B.set_span_buffer(span)
    try:
        (sd2, sp2, bd2, bp2), _ = _run_both(w, lay, x, 300, 40, chunk_in_call=True)
    finally:
        B.set_span_buffer(None)
    assert torch.equal(_bits(bd), _bits(bd2)) and torch.equal(_bits(bp), _bits(bp2))
    p0, p1, d0, d1 = span.cpu().tolist()
    assert 0 < p0 < p1 and 0 < d0 < d1, (p0, p1, d0, d1)
    assert d0 >= p0
    # off again: a further call leaves the record as it was
    before = span.clone()
    _run_both(w, lay, x, 300, 40, chunk_in_call=True)
    assert torch.equal(span, before)
