"""fp8 (E4M3) KV cache on the GPU against the oracle.

kv_append_fp8 must write the same bytes as ``oracle.fp8.kv_append`` (the
quantiser written from the E4M3 definition).  Decode over the fp8 pools is
compared with the fp64 oracle run on the dequantised pools (code value x
scale), at the bf16 tolerance 2e-2: the kernel's only roundings are the
bf16 -> f16 query, the f16 probabilities and the bf16 output."""
import numpy as np
import pytest
import torch

import gpu_cases as G
import oracle
from oracle import fp8 as F
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NAN_CODE = 0x7F


def _f32(t):
    return G.cpu(t).float().numpy()


def _pools(w, lay, layer=0, device="cpu"):
    ks, vs = W.fp8_scales(w, layer)
    kc = W.draw_fp8_pool(w, lay, ks, layer, 0, device=device)
    vc = W.draw_fp8_pool(w, lay, vs, layer, 1, device=device)
    return ks, vs, kc, vc


def _gpu_append(x, kc, vc, ks, vs, slots):
    kc, vc = kc.cuda(), vc.cuda()
    B.kv_append_fp8(x.k_new.cuda(), x.v_new.cuda(), kc, vc, ks.cuda(), vs.cuda(), slots.cuda())
    torch.cuda.synchronize()
    return kc, vc


def _oracle_append(x, kc, vc, ks, vs, slots):
    rk, rv = G.cpu(kc).numpy().copy(), G.cpu(vc).numpy().copy()
    F.kv_append(_f32(x.k_new), _f32(x.v_new), rk, rv, slots.numpy(), ks.numpy(), vs.numpy())
    return rk, rv


def _gpu_decode(w, q, kc, vc, ks, vs, bt, lens, max_seq_len=None, check_err=True):
    q = q.cuda()
    out = torch.empty_like(q)
    msl = int(lens.max()) if max_seq_len is None else max_seq_len
    ws = B.decode_workspace(q.shape[0], q.shape[1], q.shape[2], msl)
    B.paged_decode_attention_fp8(out, q, kc, vc, ks.cuda(), vs.cuda(), bt.cuda().contiguous(),
                                 lens.cuda().to(torch.int32), msl, w.scale, ws)
    torch.cuda.synchronize()
    if check_err:
        assert B.get_device_error() == 0
    return G.cpu(out)


def _oracle_decode(w, q, rk, rv, ks, vs, bt, lens, rows=None):
    """fp64 decode over the dequantised pools; ``rows`` restricts it to some
    sequences by copying just their blocks into a compact pool."""
    if rows is not None:
        blocks, nbt = [], torch.zeros(len(rows), bt.shape[1], dtype=torch.int32)
        for i, r in enumerate(rows):
            n = -(-int(lens[r]) // w.block_size)
            nbt[i, :n] = torch.arange(len(blocks), len(blocks) + n, dtype=torch.int32)
            blocks += bt[r, :n].tolist()
        idx = np.asarray(blocks)
        rk, rv, bt, lens, q = rk[idx], rv[idx], nbt, lens[rows], q[rows]
    dk = torch.from_numpy(F.dequantize_pool(rk, ks.numpy()))
    dv = torch.from_numpy(F.dequantize_pool(rv, vs.numpy()))
    return oracle.paged_decode(G.cpu(q).double(), dk, dv, bt, lens, w.scale)


@pytest.mark.parametrize("name", ["toy_decode", "llama8b_decode", "ragged_prefill"])
def test_fp8_append_bit_exact(name):
    w = W.WORKLOADS[name]
    lay = W.make_layout(w)
    dev = "cpu" if name == "toy_decode" else "cuda"
    x = W.draw_layer(w, lay, 0, device=dev, with_pool=False)
    ks, vs, kc, vc = _pools(w, lay, device=dev)
    gk, gv = _gpu_append(x, kc, vc, ks, vs, lay.slot_mapping)
    assert B.get_device_error() == 0
    rk, rv = _oracle_append(x, kc, vc, ks, vs, lay.slot_mapping)
    assert np.array_equal(G.cpu(gk).numpy(), rk)
    assert np.array_equal(G.cpu(gv).numpy(), rv)


def test_fp8_append_rounding_saturation_and_specials():
    """Exact ties (to the even mantissa), subnormal ties, values past 448,
    infinities and signed zero, at scales 1, 0.5 and 2 (exact divisions),
    and a non-power-of-two scale on random values."""
    specials = [0.0, -0.0, 1.0, 1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10,
                -(2.0 ** -10), 2.0 ** -9, 7 * 2.0 ** -10, 448.0, 450.0, 464.0, 480.0, 500.0,
                -1e4, 1e30, float("inf"), float("-inf"), 240.0, 232.0, 248.0, 0.01]
    d = 128
    row = torch.tensor((specials * (d // len(specials) + 1))[:d], dtype=torch.float32)
    g = torch.Generator().manual_seed(12)
    rnd = torch.randn(5, d, generator=g) * 3
    k_new = torch.stack([row, row * 0.5, row * 2, *rnd]).to(torch.bfloat16)   # T = 8 tokens
    t = k_new.shape[0]
    k_new = k_new[:, None, :].contiguous()
    v_new = (-k_new.float()).to(torch.bfloat16)
    nb = 4
    kc = torch.full((nb, 1, 16, d), 0x55, dtype=torch.uint8)
    vc = kc.clone()
    slots = torch.tensor([3, 20, 63, 0, 17, 40, 41, 5], dtype=torch.int64)[:t]
    for ks_val in (1.0, 0.5, 2.0, 0.0173):
        ks = torch.tensor([ks_val], dtype=torch.float32)
        vs = torch.tensor([ks_val * 2], dtype=torch.float32)
        x = W.LayerInputs(None, None, k_new, v_new, None, None)
        gk, gv = _gpu_append(x, kc, vc, ks, vs, slots)
        assert B.get_device_error() == 0
        rk, rv = _oracle_append(x, kc, vc, ks, vs, slots)
        assert np.array_equal(G.cpu(gk).numpy(), rk), ks_val
        assert np.array_equal(G.cpu(gv).numpy(), rv), ks_val


def test_fp8_append_skips_padding_and_reports_bad_slot():
    w = W.WORKLOADS["toy_decode"]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0, with_pool=False)
    ks, vs, kc, vc = _pools(w, lay)
    slots = lay.slot_mapping.clone()
    slots[2] = -1
    slots[7] = lay.num_blocks * w.block_size
    gk, gv = _gpu_append(x, kc, vc, ks, vs, slots)
    assert B.get_device_error() == 1
    keep = slots.clone()
    keep[7] = -1
    rk, rv = _oracle_append(x, kc, vc, ks, vs, keep)
    assert np.array_equal(G.cpu(gk).numpy(), rk)
    assert np.array_equal(G.cpu(gv).numpy(), rv)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 8), (16, 2), (16, 1)])
def test_fp8_decode_edge_lengths_and_groups(hq, hkv):
    """Block (16), stage (64) and split (512) boundaries, one token, every
    compiled group size; NaN codes in every pool row no sequence uses."""
    w = G.custom_workload(torch.bfloat16, hq, hkv, 128, seed=41)
    lens = [1, 2, 15, 16, 17, 33, 63, 64, 65, 511, 512, 513, 1024, 1025, 1600]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0, with_pool=False)
    ks, vs, kc, vc = _pools(w, lay)
    unused = ~G.used_slot_mask(lay, w.block_size)
    kc.permute(0, 2, 1, 3)[unused] = NAN_CODE
    vc.permute(0, 2, 1, 3)[unused] = NAN_CODE
    gk, gv = _gpu_append(x, kc, vc, ks, vs, lay.slot_mapping)
    rk, rv = _oracle_append(x, kc, vc, ks, vs, lay.slot_mapping)
    assert np.array_equal(G.cpu(gk).numpy(), rk) and np.array_equal(G.cpu(gv).numpy(), rv)
    got = _gpu_decode(w, x.q_decode, gk, gv, ks, vs, lay.decode_block_table, lay.seq_lens)
    ref = _oracle_decode(w, x.q_decode, rk, rv, ks, vs, lay.decode_block_table, lay.seq_lens)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= 2e-2


def test_fp8_decode_balanced_walk_nan_in_unused_rows():
    """48 seeded lengths in [1, 3000] (with 1, 64, 65, 512, 513): enough
    64-token stages for the balanced walk, which cuts sequences between CTAs
    at arbitrary stage boundaries; every output against the oracle, NaN codes
    in every unused pool row."""
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=42)
    g = torch.Generator().manual_seed(9)
    lens = torch.randint(1, 3001, (48,), generator=g).tolist()
    lens[:5] = [1, 64, 65, 512, 513]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0, with_pool=False)
    ks, vs, kc, vc = _pools(w, lay)
    unused = ~G.used_slot_mask(lay, w.block_size)
    kc.permute(0, 2, 1, 3)[unused] = NAN_CODE
    vc.permute(0, 2, 1, 3)[unused] = NAN_CODE
    gk, gv = _gpu_append(x, kc, vc, ks, vs, lay.slot_mapping)
    rk, rv = _oracle_append(x, kc, vc, ks, vs, lay.slot_mapping)
    assert np.array_equal(G.cpu(gk).numpy(), rk) and np.array_equal(G.cpu(gv).numpy(), rv)
    got = _gpu_decode(w, x.q_decode, gk, gv, ks, vs, lay.decode_block_table, lay.seq_lens)
    ref = _oracle_decode(w, x.q_decode, rk, rv, ks, vs, lay.decode_block_table, lay.seq_lens)
    assert torch.isfinite(got).all()
    assert G.max_err(got, ref) <= 2e-2


@pytest.mark.parametrize("name", ["llama8b_decode", "ragged_prefill"])
def test_fp8_decode_full_size_sampled_sequences(name):
    """One full-size layer in the launch configuration of the step; every
    head of 10 sampled sequences (the longest and shortest among them)."""
    w = W.WORKLOADS[name]
    lay = W.make_layout(w)
    x = W.draw_layer(w, lay, 0, device="cuda", with_pool=False)
    ks, vs, kc, vc = _pools(w, lay, device="cuda")
    gk, gv = _gpu_append(x, kc, vc, ks, vs, lay.slot_mapping)
    got = _gpu_decode(w, x.q_decode, gk, gv, ks, vs, lay.decode_block_table, lay.seq_lens)
    lens = lay.seq_lens
    g = torch.Generator().manual_seed(77)
    rows = sorted({int(lens.argmax()), int(lens.argmin()),
                   *torch.randperm(w.num_seqs, generator=g)[:8].tolist()})
    ref = _oracle_decode(w, x.q_decode, G.cpu(gk).numpy(), G.cpu(gv).numpy(), ks, vs,
                         lay.decode_block_table, lens, rows=rows)
    assert G.max_err(got[rows], ref) <= 2e-2


def test_fp8_decode_quantisation_error_is_bounded():
    """Property at any size: decode over the fp8 cache stays close to decode
    over the bf16 values it quantised (E4M3 keeps 3 mantissa bits: relative
    error at most 2^-4 per element before saturation)."""
    w = G.custom_workload(torch.bfloat16, 32, 8, 128, seed=5)
    lens = [300, 2000, 77]
    lay = W.make_layout(w, seq_lens_after=lens, prefill=(0, 0))
    x = W.draw_layer(w, lay, 0)
    ks = torch.full((8,), 6.0 / 448.0)
    vs = torch.full((8,), 6.0 / 448.0)
    kc8 = torch.zeros(lay.num_blocks, 8, 16, 128, dtype=torch.uint8)
    vc8 = torch.zeros_like(kc8)
    kb = torch.zeros(lay.num_blocks, 8, 16, 128, dtype=torch.bfloat16)
    vb = torch.zeros_like(kb)
    # fill every used slot from bf16 values, through both appends
    slots, kk, vv = [], [], []
    gen = torch.Generator().manual_seed(6)
    for b, n in enumerate(lens):
        for p in range(n):
            slots.append(int(lay.block_table[b, p // 16]) * 16 + p % 16)
    slots = torch.tensor(slots, dtype=torch.int64)
    kk = torch.randn(len(slots), 8, 128, generator=gen).to(torch.bfloat16)
    vv = torch.randn(len(slots), 8, 128, generator=gen).to(torch.bfloat16)
    xx = W.LayerInputs(None, None, kk, vv, None, None)
    gk, gv = _gpu_append(xx, kc8, vc8, ks, vs, slots)
    gkb, gvb = kb.cuda(), vb.cuda()
    B.kv_append(kk.cuda(), vv.cuda(), gkb, gvb, slots.cuda())
    q = x.q_decode
    o8 = _gpu_decode(w, q, gk, gv, ks, vs, lay.decode_block_table, lay.seq_lens)
    o16 = G.gpu_decode(w, q, gkb, gvb, lay.decode_block_table, lay.seq_lens)
    ref16 = oracle.paged_decode(q, G.cpu(gkb), G.cpu(gvb), lay.decode_block_table, lay.seq_lens,
                                w.scale)
    assert G.max_err(o16, ref16) <= 2e-2
    assert G.max_err(o8, ref16) <= 0.05


def test_fp8_decode_rejects_unsupported_and_missing_scales():
    w = G.custom_workload(torch.bfloat16, 8, 2, 64, seed=3)
    lay = W.make_layout(w, seq_lens_after=[5], prefill=(0, 0))
    kc = torch.zeros(lay.num_blocks, 2, 16, 64, dtype=torch.uint8, device="cuda")
    q = torch.zeros(1, 8, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.ones(2, device="cuda")
    with pytest.raises(B.PagedKVError) as e:
        B.paged_decode_attention_fp8(torch.empty_like(q), q, kc, kc, s, s,
                                     lay.decode_block_table.cuda(), lay.seq_lens.cuda(), 5, w.scale)
    assert e.value.status == 5          # head_dim 64: unsupported
    w = G.custom_workload(torch.bfloat16, 8, 2, 128, seed=3)
    kc = torch.zeros(lay.num_blocks, 2, 16, 128, dtype=torch.uint8, device="cuda")
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PagedKVError) as e:
        B.paged_decode_attention_fp8(torch.empty_like(q), q, kc, kc, None, s,
                                     lay.decode_block_table.cuda(), lay.seq_lens.cuda(), 5, w.scale,
                                     B.decode_workspace(1, 8, 128, 5))
    assert e.value.status == 1          # no K scale
