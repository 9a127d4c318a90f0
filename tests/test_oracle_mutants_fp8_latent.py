"""Planted mistakes in copies of the fp8 and latent-cache oracles must be
caught by their pins (CPU only).  Each mutant is a plausible slip in
oracle/fp8.py or oracle/mla.py; at least one check must fail for it."""
import math

import numpy as np
import pytest
import torch

from oracle import fp8 as F
from oracle import mla as M
from paged_kv_cache_104_gb300 import workloads as W


# ---------------------------------------------------------------- fp8
def _fp8_checks(encode, decode_table):
    """The pins of tests/test_fp8_oracle.py, parameterised by the functions."""
    t = decode_table()
    assert t[0x38] == 1.0 and t[0xC0] == -2.0 and t[0x7E] == 448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6
    cases = {1.0625: 0x38, 1.1875: 0x3A, 2.0 ** -10: 0x00, 3 * 2.0 ** -11: 0x01,
             464.0: 0x7E, 500.0: 0x7E, -1e30: 0xFE, -0.0: 0x80}
    for y, code in cases.items():
        assert int(encode([y])[0]) == code, y
    g = torch.Generator().manual_seed(3)
    y = (torch.randn(5000, generator=g) * 10)
    y = y[y.abs() < 464]
    assert np.array_equal(encode(y.double().numpy()), y.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def _encode_mutant(kind):
    def enc(y):
        y = np.asarray(y, dtype=np.float64)
        a, neg = np.abs(y), np.signbit(y)
        if kind != "no_saturation":
            a = np.minimum(a, 448.0)
        pos = F.decode_table()[:127]
        hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 126)
        lo = np.clip(hi - 1, 0, 126)
        dh, dl = np.abs(pos[hi] - a), np.abs(a - pos[lo])
        if kind == "round_half_up":
            pick_lo = dl < dh
        elif kind == "truncate":
            pick_lo = pos[hi] > a
        else:   # ties away from zero
            pick_lo = dl < dh
            pick_lo = np.where(dl == dh, False, pick_lo)
        code = np.where(pick_lo, lo, hi).astype(np.uint8)
        if kind == "no_saturation":
            code = np.where(a > 448.0, 0x7F, code).astype(np.uint8)
        return (code | np.where(neg, 0x80, 0).astype(np.uint8)).astype(np.uint8)
    return enc


def _table_mutant_bias8():
    t = F.decode_table().copy()
    for code in range(256):
        e, m = (code >> 3) & 0xF, code & 7
        if 0 < e < 15 or (e == 15 and m != 7):
            s = -1.0 if code & 0x80 else 1.0
            t[code] = s * (1 + m / 8) * 2.0 ** (e - 8)
    return lambda: t


def test_fp8_oracle_passes_its_pins():
    _fp8_checks(F.encode, F.decode_table)


@pytest.mark.parametrize("kind", ["round_half_up", "truncate", "ties_away", "no_saturation"])
def test_fp8_encode_mutants_are_caught(kind):
    with pytest.raises(AssertionError):
        _fp8_checks(_encode_mutant(kind), F.decode_table)


def test_fp8_decode_bias_mutant_is_caught():
    with pytest.raises(AssertionError):
        _fp8_checks(F.encode, _table_mutant_bias8())


# ---------------------------------------------------------------- latent cache
def _mla_mutant(kind):
    def decode(q, w_k, w_v, pool, block_table, seq_lens, scale, seqs=None):
        if kind == "swap_projections":
            return M.mla_decode(q, w_v, w_k, pool, block_table, seq_lens, scale, seqs)
        if kind == "transpose_wk":
            return M.mla_decode(q, w_k.transpose(1, 2).contiguous(), w_v, pool, block_table,
                                seq_lens, scale, seqs)
        # values taken from the latent directly (no W_V), keys as they should be
        seqs = range(q.shape[0]) if seqs is None else seqs
        outs = []
        for b in seqs:
            n = int(seq_lens[b])
            c = M.gather_latents(pool, block_table[b], n)
            o = torch.empty(q.shape[1], q.shape[2], dtype=torch.float64)
            for h in range(q.shape[1]):
                k = c @ w_k[h].to(torch.float64).T
                s = (k @ q[b, h].to(torch.float64)) * scale
                p = torch.softmax(s, 0)
                o[h] = (p @ c)[: q.shape[2]]
            outs.append(o)
        return torch.stack(outs)
    return decode


def _mla_checks(decode):
    """Brute force with random square projections and the one-token closed
    form (the pins of tests/test_mla_oracle.py)."""
    from test_mla_oracle import _brute, _layout, _pool
    lens = [3, 18]
    hq, d, r = 2, 6, 6
    w, lay = _layout(lens, hq, r, seed=5)
    pool = _pool(lay, r, 6)
    g = torch.Generator().manual_seed(7)
    q = torch.randn(2, hq, d, generator=g, dtype=torch.float64)
    wk = torch.randn(hq, d, r, generator=g, dtype=torch.float64)
    wv = torch.randn(hq, d, r, generator=g, dtype=torch.float64)
    got = decode(q, wk, wv, pool, lay.block_table, lay.seq_lens, 0.41)
    ref = _brute(q, wk, wv, pool, lay.block_table, lay.seq_lens, 0.41)
    assert torch.allclose(got, ref, atol=1e-12, rtol=0)


def test_mla_oracle_passes_its_pins():
    _mla_checks(M.mla_decode)


@pytest.mark.parametrize("kind", ["swap_projections", "transpose_wk", "value_without_projection"])
def test_mla_mutants_are_caught(kind):
    with pytest.raises(AssertionError):
        _mla_checks(_mla_mutant(kind))
