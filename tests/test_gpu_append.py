"""kv_append on the GPU: bit-exact against the oracle's scatter, every other
byte of the pools untouched, padding slots skipped, bad slots reported."""
import pytest
import torch

import gpu_cases as G
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("name", ["tiny_fp32", "toy_decode", "llama8b_decode", "ragged_prefill",
                                  "long_context"])
def test_append_bit_exact(name):
    w = W.WORKLOADS[name]
    lay = W.make_layout(w)
    dev = "cpu" if name in ("tiny_fp32", "toy_decode") else "cuda"
    x = W.draw_layer(w, lay, 0, device=dev)
    kc, vc = G.gpu_append(lay, x)
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    rk, rv = G.oracle_append(lay, x)
    assert torch.equal(_bits(G.cpu(kc)), _bits(rk))
    assert torch.equal(_bits(G.cpu(vc)), _bits(rv))


def test_append_skips_padding_and_reports_bad_slot():
    w = W.WORKLOADS["toy_decode"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0)
    slots = lay.slot_mapping.clone()
    slots[3] = -1                                   # padding
    slots[5] = lay.num_blocks * w.block_size        # one past the pool
    kc, vc = x.k_cache.cuda(), x.v_cache.cuda()
    B.kv_append(x.k_new.cuda(), x.v_new.cuda(), kc, vc, slots.cuda())
    torch.cuda.synchronize()
    assert B.get_device_error() == 1
    assert B.get_device_error() == 0                # cleared
    keep = slots.clone()
    keep[5] = -1
    rk, rv = G.oracle_append(lay, x, slots=keep)
    assert torch.equal(_bits(G.cpu(kc)), _bits(rk))
    assert torch.equal(_bits(G.cpu(vc)), _bits(rv))


def test_append_empty_is_noop():
    w = W.WORKLOADS["tiny_fp32"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0)
    kc = x.k_cache.cuda()
    before = kc.clone()
    B.kv_append(x.k_new[:0].cuda(), x.v_new[:0].cuda(), kc, kc.clone(),
                lay.slot_mapping[:0].cuda())
    torch.cuda.synchronize()
    assert torch.equal(_bits(kc), _bits(before))
