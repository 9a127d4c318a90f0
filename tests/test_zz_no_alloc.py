"""The allocation-free decode entry point, through the C ABI.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate device
memory for a workspace (an engine that owns all device memory in its own pool
and forbids later allocations, or a plugin interface that passes only input
and output pointers).  It keeps its split partials in a scratch array inside
the library.

The test makes three calls in a row, each with other lengths and inputs, so
stale scratch contents from an earlier call would show:
  * 64 sequences at 2,301 tokens -- large enough for the balanced walk, whose
    per-stream partial counts live in the scratch array too;
  * a ragged batch of 7 sequences (512-token splits);
  * a ragged batch of 4 sequences.
Each output must equal, bit for bit, the ordinary entry point's with a
workspace (the same kernels walk the same plan) and must be within the bf16
tolerance of the fp64 oracle.  A size beyond the scratch array is refused
before any launch.

The file is named so that pytest collects it after every other test file.
"""
import pytest
import torch

import gpu_cases as G
import oracle
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _ragged_case(lens, seed):
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=seed)
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    return w, lay, W.draw_layer(w, lay, 0)


def _balanced_case():
    w = W.WORKLOADS["llama8b_decode"]
    lay = W.make_layout(w)
    return w, lay, W.draw_layer(w, lay, 0, device="cuda")


def _run_case(w, lay, x):
    kc, vc = G.gpu_append(lay, x)
    q = x.q_decode.cuda()
    bt = lay.decode_block_table.cuda().contiguous()
    sl = lay.seq_lens.cuda()
    msl = int(lay.seq_lens.max())
    assert 0 < B.decode_workspace_bytes(q.shape[0], 32, 128, msl) <= B.NOALLOC_SCRATCH_BYTES
    ref = torch.empty_like(q)
    ws = B.decode_workspace(q.shape[0], 32, 128, msl)
    B.paged_decode_attention(ref, q, kc, vc, bt, sl, msl, w.scale, ws)
    got = torch.full_like(q, float("nan"))
    B.paged_decode_attention_noalloc(got, q, kc, vc, bt, sl, msl, w.scale)
    torch.cuda.synchronize()
    assert B.get_device_error() == 0
    rk, rv = G.oracle_append(lay, x)
    want = oracle.paged_decode(G.cpu(x.q_decode), rk, rv, lay.decode_block_table, lay.seq_lens,
                               w.scale)
    return got.cpu(), ref.cpu(), want


def test_noalloc_matches_workspace_path_and_oracle_on_three_calls():
    cases = [_balanced_case(), _ragged_case([3000, 17, 1200, 513, 2048, 1, 4096], seed=41),
             _ragged_case([700, 2500, 64, 1537], seed=42)]
    for w, lay, x in cases:
        got, ref, want = _run_case(w, lay, x)
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref), "noalloc output differs from the workspace path"
        assert G.max_err(got, want) <= G.TOL[torch.bfloat16]


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
