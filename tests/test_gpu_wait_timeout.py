"""Bounded waits: a wait that runs out is reported, and the GPU stays usable.

Every mbarrier wait in the kernels gives up after a limit, records
PKV_DEVERR_TIMEOUT in the device error word and lets the kernel return
instead of hanging or trapping.  The shipped library's limit is about a
second and no correct input reaches it, so this test uses a test-only build
(``build.build_wait_test``): the decode kernel compiled with its wait limit
cut to about 2 ms and its producer withholding every copy.  The consumers'
first waits then run out with no copy in flight.  The test checks that the
call returns, that the error word of that build reads PKV_DEVERR_TIMEOUT,
and that the shipped library, run next on the same GPU and inputs, still
matches the oracle.
"""
import ctypes

import pytest
import torch

import gpu_cases as G
import oracle
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import build as BL
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PKV_DEVERR_TIMEOUT = 4


def test_decode_wait_time_out_is_reported_and_gpu_stays_usable():
    lib = B.open_library(BL.build_wait_test())
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=5)
    lay = W.make_layout(w, seq_lens_after=[700, 33, 1500, 64], prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    kc, vc = G.gpu_append(lay, x)
    q = x.q_decode.cuda()
    bt = lay.decode_block_table.cuda().contiguous()
    sl = lay.seq_lens.cuda()
    msl = int(lay.seq_lens.max())
    ws = B.decode_workspace(q.shape[0], 32, 128, msl)
    out = torch.zeros_like(q)

    code = ctypes.c_int(-1)
    assert lib.pkv_get_device_error(ctypes.byref(code), 1) == 0
    assert code.value == 0
    st = lib.pkv_paged_decode_attention(
        out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), sl.data_ptr(),
        q.shape[0], bt.shape[1], msl, kc.shape[0], 32, 8, 128, 16, w.scale, ws.data_ptr(),
        ws.numel(), B.PKV_BF16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert lib.pkv_get_device_error(ctypes.byref(code), 1) == 0
    assert code.value == PKV_DEVERR_TIMEOUT

    # the same GPU, the shipped library, the same inputs: correct results
    got = G.gpu_decode(w, x.q_decode, kc, vc, lay.decode_block_table, lay.seq_lens)
    rk, rv = G.oracle_append(lay, x)
    want = oracle.paged_decode(G.cpu(x.q_decode), rk, rv, lay.decode_block_table, lay.seq_lens,
                               w.scale)
    assert G.max_err(got, want) <= G.TOL[torch.bfloat16]
    assert B.get_device_error() == 0
