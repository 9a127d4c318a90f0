"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs."""
from __future__ import annotations

import torch

import oracle
from paged_kv_cache_104_gb300 import binding as B
from paged_kv_cache_104_gb300 import workloads as W

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


def cpu(t):
    return t.detach().to("cpu")


def used_slot_mask(lay: W.Layout, bs: int, prefill_len: int = 0) -> torch.Tensor:
    """[num_blocks, bs] True where some sequence stores a token (the decode
    rows up to seq_lens, and the prefill row up to ``prefill_len``)."""
    m = torch.zeros(lay.num_blocks, bs, dtype=torch.bool)
    rows = list(enumerate(lay.seq_lens.tolist()))
    if lay.prefill_row >= 0 and prefill_len:
        rows.append((lay.prefill_row, prefill_len))
    for r, n in rows:
        for j in range(-(-n // bs)):
            blk = int(lay.block_table[r, j])
            m[blk, : min(bs, n - j * bs)] = True
    return m


def poison_unused(kc: torch.Tensor, vc: torch.Tensor, mask: torch.Tensor) -> None:
    """Fill every pool row no sequence uses with NaN (in place)."""
    bad = ~mask
    kc.permute(0, 2, 1, 3)[bad] = float("nan")
    vc.permute(0, 2, 1, 3)[bad] = float("nan")


def gpu_append(lay, x, dev="cuda"):
    kc, vc = x.k_cache.to(dev), x.v_cache.to(dev)
    B.kv_append(x.k_new.to(dev), x.v_new.to(dev), kc, vc, lay.slot_mapping.to(dev))
    return kc, vc


def oracle_append(lay, x, slots=None):
    kc, vc = cpu(x.k_cache).clone(), cpu(x.v_cache).clone()
    oracle.kv_append(cpu(x.k_new), cpu(x.v_new), kc, vc, lay.slot_mapping if slots is None else slots)
    return kc, vc


def gpu_decode(w, q, kc, vc, block_table, seq_lens, max_seq_len=None, check_err=True):
    dev = kc.device
    q = q.to(dev)
    out = torch.empty_like(q)
    bt = block_table.to(dev).contiguous()
    sl = seq_lens.to(dev).to(torch.int32)
    msl = int(seq_lens.max()) if max_seq_len is None else max_seq_len
    ws = B.decode_workspace(q.shape[0], q.shape[1], q.shape[2], msl, device=dev)
    B.paged_decode_attention(out, q, kc, vc, bt, sl, msl, w.scale, ws)
    torch.cuda.synchronize()
    if check_err:
        assert B.get_device_error() == 0
    return out


def gpu_prefill(w, q, kc, vc, bt_row, prior, check_err=True):
    dev = kc.device
    q = q.to(dev)
    out = torch.empty_like(q)
    B.chunked_prefill_attention(out, q, kc, vc, bt_row.to(dev).contiguous(), prior, w.scale)
    torch.cuda.synchronize()
    if check_err:
        assert B.get_device_error() == 0
    return out


def max_err(got: torch.Tensor, ref: torch.Tensor) -> float:
    return float((cpu(got).double() - ref.double()).abs().max())


def custom_workload(dtype, hq, hkv, d, seed=7, name="custom"):
    return W.Workload(name, dtype, 1, hq, hkv, d, 16, 1, seed=seed, context=(1,))
