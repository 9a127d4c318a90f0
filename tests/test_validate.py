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
