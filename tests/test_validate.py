"""The binding's debug mode: host-side checks of slots, block tables and
lengths before a call (no GPU needed).  Good index arrays pass; each kind of
bad entry raises PagedKVError with PKV_EINVAL before the library is touched."""
import pytest
import torch

from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import validate as V
from paged_kv_cache_104_gb300 import workloads as W

import gpu_cases as G


def _layout():
    w = G.custom_workload(torch.bfloat16, 8, 2, 128, seed=7)
    return w, W.make_layout(w, seq_lens_after=[1, 17, 300], prefill=(40, 70))


def test_good_arrays_pass():
    w, lay = _layout()
    V.check_slots(lay.slot_mapping, lay.num_blocks, 16)
    V.check_decode(lay.decode_block_table, lay.seq_lens, int(lay.seq_lens.max()),
                   lay.num_blocks, 16, appends=True)
    V.check_prefill(lay.block_table[lay.prefill_row], 40, 70, lay.num_blocks, 16)
    V.check_slots(torch.tensor([-1, -1, 5]), 1, 16)          # negative slots are padding


@pytest.mark.parametrize("slots,match", [
    ([0, 3, 3], "more than once"),
    ([0, 16 * 4], "outside the pool"),
])
def test_bad_slots(slots, match):
    with pytest.raises(V.ValidationError, match=match):
        V.check_slots(torch.tensor(slots, dtype=torch.int64), 4, 16)


def test_bad_lengths_and_blocks():
    w, lay = _layout()
    bt, lens = lay.decode_block_table.clone(), lay.seq_lens.clone()
    msl = int(lens.max())
    with pytest.raises(V.ValidationError, match="seq_lens"):
        V.check_decode(bt, torch.tensor([0, 17, 300], dtype=torch.int32), msl, lay.num_blocks, 16)
    with pytest.raises(V.ValidationError, match="seq_lens"):
        V.check_decode(bt, lens, 100, lay.num_blocks, 16)     # 300 > max_seq_len
    bad = bt.clone()
    bad[2, 5] = lay.num_blocks
    with pytest.raises(V.ValidationError, match="block_table"):
        V.check_decode(bad, lens, msl, lay.num_blocks, 16)
    bad = bt.clone()
    bad[0, 5] = -3                                             # row 0 holds one token: unused
    V.check_decode(bad, lens, msl, lay.num_blocks, 16)
    shared = bt.clone()
    shared[1, 1] = shared[2, 18]                               # both new tokens in one row
    lens2 = torch.tensor([1, 17, 289], dtype=torch.int32)
    with pytest.raises(V.ValidationError, match="more than once"):
        V.check_decode(shared, lens2, msl, lay.num_blocks, 16, appends=True)
    row = lay.block_table[lay.prefill_row].clone()
    row[3] = -1
    with pytest.raises(V.ValidationError, match="prefill block table"):
        V.check_prefill(row, 40, 70, lay.num_blocks, 16)
    with pytest.raises(V.ValidationError, match="need"):
        V.check_prefill(row[:2], 40, 70, lay.num_blocks, 16)


def test_debug_mode_raises_before_the_library(monkeypatch):
    """With debug mode on, a bad call raises PagedKVError (PKV_EINVAL) from the
    host check; the library is never loaded for it."""
    w, lay = _layout()
    def no_library():
        raise AssertionError("the library was reached")
    monkeypatch.setattr(B, "load", no_library)
    B.set_debug(True)
    try:
        x = W.draw_layer(w, lay, 0)
        slots = lay.slot_mapping.clone()
        slots[1] = slots[0]
        with pytest.raises(B.PagedKVError) as e:
            B.kv_append(x.k_new, x.v_new, x.k_cache, x.v_cache, slots)
        assert e.value.status == 1 and "more than once" in str(e.value)
        lens = lay.seq_lens.clone()
        lens[0] = 0
        with pytest.raises(B.PagedKVError) as e:
            B.paged_decode_attention(torch.empty_like(x.q_decode), x.q_decode, x.k_cache,
                                     x.v_cache, lay.decode_block_table, lens, 300, w.scale)
        assert e.value.status == 1
    finally:
        B.set_debug(False)


def _small():
    """4 blocks of 16 rows, 2 KV heads, head_dim 8, 4 query heads (CPU)."""
    nb, hkv, bs, d, hq = 4, 2, 16, 8, 4
    bf = torch.bfloat16
    t = dict(
        kc=torch.zeros(nb, hkv, bs, d, dtype=bf), vc=torch.zeros(nb, hkv, bs, d, dtype=bf),
        kc8=torch.zeros(nb, hkv, bs, d, dtype=torch.uint8),
        vc8=torch.zeros(nb, hkv, bs, d, dtype=torch.uint8),
        sc=torch.ones(hkv), k_new=torch.zeros(2, hkv, d, dtype=bf),
        v_new=torch.zeros(2, hkv, d, dtype=bf), q=torch.zeros(2, hq, d, dtype=bf),
        out=torch.zeros(2, hq, d, dtype=bf),
        bt=torch.tensor([[0, 1], [2, 3]], dtype=torch.int32),
        lens=torch.tensor([5, 20], dtype=torch.int32),
        c_cache=torch.zeros(nb, bs, d, dtype=bf), c_new=torch.zeros(2, d, dtype=bf),
        w=torch.zeros(hq, d, d, dtype=bf))
    return t


def _calls():
    """(name, call, message) with one bad entry each."""
    i32 = lambda v: torch.tensor(v, dtype=torch.int32)
    i64 = lambda v: torch.tensor(v, dtype=torch.int64)
    same_row = i32([[0, 1], [0, 1]]), i32([17, 17])   # both new tokens at block 1, row 0
    return [
        ("kv_append_fp8", lambda t: B.kv_append_fp8(t["k_new"], t["v_new"], t["kc8"], t["vc8"],
                                                     t["sc"], t["sc"], i64([3, 3])), "more than once"),
        ("latent_append", lambda t: B.latent_append(t["c_new"], t["c_cache"], i64([0, 64])),
         "outside the pool"),
        ("paged_decode_attention_fp8",
         lambda t: B.paged_decode_attention_fp8(t["out"], t["q"], t["kc8"], t["vc8"], t["sc"],
                                                t["sc"], i32([[0, 1], [2, 9]]), t["lens"], 32, 1.0),
         "block_table"),
        ("mla_decode_attention (appending)",
         lambda t: B.mla_decode_attention(t["out"], t["q"], t["w"], t["w"], t["c_cache"],
                                          same_row[0], same_row[1], 32, 1.0, c_new=t["c_new"]),
         "more than once"),
        ("paged_decode_attention_noalloc",
         lambda t: B.paged_decode_attention_noalloc(t["out"], t["q"], t["kc"], t["vc"], t["bt"],
                                                    i32([5, 40]), 32, 1.0), "seq_lens"),
        ("paged_decode_attention_append",
         lambda t: B.paged_decode_attention_append(t["out"], t["q"], t["k_new"], t["v_new"], t["kc"],
                                                   t["vc"], same_row[0], same_row[1], 32, 1.0),
         "more than once"),
        ("chunked_prefill_attention",
         lambda t: B.chunked_prefill_attention(torch.zeros(20, 4, 8, dtype=torch.bfloat16),
                                               torch.zeros(20, 4, 8, dtype=torch.bfloat16),
                                               t["kc"], t["vc"], i32([0]), 0, 1.0), "need"),
        ("decode_prefill_attention (chunk slots)",
         lambda t: B.decode_prefill_attention(
             t["out"], t["q"], t["k_new"], t["v_new"], t["kc"], t["vc"], t["bt"], t["lens"], 32,
             torch.zeros(2, 4, 8, dtype=torch.bfloat16), torch.zeros(2, 4, 8, dtype=torch.bfloat16),
             i32([3]), 0, 1.0, chunk_k_new=t["k_new"], chunk_v_new=t["v_new"],
             chunk_slots=i64([0, 99])), "outside the pool"),
    ]


@pytest.mark.parametrize("case", range(len(_calls())), ids=[c[0] for c in _calls()])
def test_debug_mode_covers_every_wrapper(case, monkeypatch):
    """Each wrapper runs its host checks in debug mode and raises PKV_EINVAL
    for a bad entry without reaching the library."""
    name, call, match = _calls()[case]
    def no_library():
        raise AssertionError("the library was reached")
    monkeypatch.setattr(B, "load", no_library)
    B.set_debug(True)
    try:
        with pytest.raises(B.PagedKVError, match=match) as e:
            call(_small())
        assert e.value.status == 1
    finally:
        B.set_debug(False)


def test_debug_mode_lets_good_calls_through(monkeypatch):
    """Valid index arrays pass the host checks: the call goes on to the
    library (stubbed here to stop it)."""
    class Reached(Exception):
        pass
    def stub():
        raise Reached
    monkeypatch.setattr(B, "load", stub)
    t = _small()
    B.set_debug(True)
    try:
        with pytest.raises(Reached):
            B.paged_decode_attention_append(t["out"], t["q"], t["k_new"], t["v_new"], t["kc"],
                                            t["vc"], t["bt"], t["lens"], 32, 1.0)
        with pytest.raises(Reached):
            B.kv_append_fp8(t["k_new"], t["v_new"], t["kc8"], t["vc8"], t["sc"], t["sc"],
                            torch.tensor([3, 20], dtype=torch.int64))
        with pytest.raises(Reached):
            B.chunked_prefill_attention(torch.zeros(20, 4, 8, dtype=torch.bfloat16),
                                        torch.zeros(20, 4, 8, dtype=torch.bfloat16),
                                        t["kc"], t["vc"], torch.tensor([0, 1], dtype=torch.int32),
                                        0, 1.0)
    finally:
        B.set_debug(False)
