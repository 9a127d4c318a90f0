"""The allocation-free decode entry point, through the C ABI.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate device
memory for a workspace (an engine that owns all device memory in its own pool
and forbids later allocations, or a plugin interface that passes only input
and output pointers).  It keeps its split partials in a scratch array inside
the library.  This test checks that two calls in a row -- the second with
other lengths and inputs, so stale scratch contents from the first would
show -- give the same output as the ordinary entry point with a workspace,
and that a size beyond the scratch array is refused before any launch.

The file is named so that pytest collects it after every other test file.
"""
import pytest
import torch

import gpu_cases as G
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _case(lens, seed):
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=seed)
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    kc, vc = G.gpu_append(lay, x)
    return w, lay, x, kc, vc


def _run_both(w, lay, x, kc, vc):
    q = x.q_decode.cuda()
    bt = lay.decode_block_table.cuda().contiguous()
    sl = lay.seq_lens.cuda()
    msl = int(lay.seq_lens.max())
    ref = torch.empty_like(q)
    ws = B.decode_workspace(q.shape[0], 32, 128, msl)
    B.paged_decode_attention(ref, q, kc, vc, bt, sl, msl, w.scale, ws)
    got = torch.full_like(q, float("nan"))
    B.paged_decode_attention_noalloc(got, q, kc, vc, bt, sl, msl, w.scale)
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    return got.cpu(), ref.cpu()


def test_noalloc_matches_workspace_path_on_two_calls():
    first = _case([3000, 17, 1200, 513, 2048, 1, 4096], seed=41)
    got1, ref1 = _run_both(*first)
    assert B.decode_workspace_bytes(7, 32, 128, 4096) > 0  # the scratch is really used
    second = _case([700, 2500, 64, 1537], seed=42)
    got2, ref2 = _run_both(*second)
    for got, ref in ((got1, ref1), (got2, ref2)):
        assert torch.isfinite(got).all()
        assert float((got.double() - ref.double()).abs().max()) <= 2e-2


def test_noalloc_refuses_sizes_beyond_its_scratch():
    # 8192 sequences x 32 heads x 64 splits of partials exceed the scratch array
    assert B.decode_workspace_bytes(8192, 32, 128, 32768) > B.NOALLOC_SCRATCH_BYTES
    lib = B.load()
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    st = lib.pkv_paged_decode_attention_noalloc(p, p, p, p, p, p, 8192, 2048, 32768, 1, 32, 8,
                                                128, 16, 0.088, 1, None)
    assert st == 3
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
