"""The E4M3 oracle against the OCP FP8 definition, a library cast, and the
rounding error bound (CPU only)."""
import math

import numpy as np
import torch

import oracle
from oracle import fp8 as F


def test_codes_from_the_definition():
    t = F.decode_table()
    assert t[0x00] == 0.0 and math.copysign(1, t[0x80]) == -1.0
    assert t[0x38] == 1.0 and t[0xC0] == -2.0
    assert t[0x08] == 2.0 ** -6           # smallest normal
    assert t[0x01] == 2.0 ** -9           # smallest subnormal
    assert t[0x07] == 7 / 8 * 2.0 ** -6   # largest subnormal
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isfinite(t).sum() == 254


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(F.encode(F.decode(codes)), codes)


def test_ties_to_even_and_saturation():
    cases = {1.0625: 0x38, 1.1875: 0x3A, 2.0 ** -10: 0x00, 3 * 2.0 ** -11: 0x01,
             464.0: 0x7E, 500.0: 0x7E, 1e30: 0x7E, -1e30: 0xFE, -0.0: 0x80}
    for y, code in cases.items():
        assert int(F.encode([y])[0]) == code, y


def test_matches_torch_cast_below_the_overflow_boundary():
    g = torch.Generator().manual_seed(3)
    y = torch.cat([torch.randn(20000, generator=g) * 10,
                   torch.randn(5000, generator=g) * 1e-2,
                   (torch.rand(5000, generator=g) - 0.5) * 900])
    y = y[y.abs() < 464]
    ours = F.encode(y.double().numpy())
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_rounding_error_bound():
    g = torch.Generator().manual_seed(4)
    y = (torch.randn(50000, generator=g) * 30).double().numpy()
    y = y[np.abs(y) >= 2.0 ** -6]
    y = np.clip(y, -448, 448)
    back = F.decode(F.encode(y))
    assert np.all(np.abs(back - y) <= np.abs(y) * 2.0 ** -4 + 1e-300)


def test_fp64_storage_reproduces_fp32_pools():
    """Dequantised pools passed as fp64 give the same attention as an fp32 pool
    of the same (exactly representable) values."""
    import oracle_pins as P
    w = P._small_workload()
    g = torch.Generator().manual_seed(5)
    k = [torch.randn(40, 2, 16, generator=g)]
    v = [torch.randn(40, 2, 16, generator=g)]
    kc, vc, lay = P._paged_from_contiguous(oracle, k, v, w)
    q = torch.randn(1, 4, 16, generator=g)
    a = oracle.paged_decode(q, kc, vc, lay.block_table, lay.seq_lens, w.scale)
    b = oracle.paged_decode(q.double(), kc.double(), vc.double(), lay.block_table, lay.seq_lens, w.scale)
    assert torch.equal(a, b)
