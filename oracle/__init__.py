"""fp64 CPU oracle for attention over a block-paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``paged_kv_cache_104_gb300``) never imports it, and this package never
imports the product path: the two share no code.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64, OpenMP over
independent (sequence, head) pairs); this module compiles it with gcc on
first use and marshals torch CPU tensors into it.  ``kv_bytes_per_token`` is
the size formula printed on "The KV cache and prefix caching", section "What
prefill stores and decode reads" (also "KV cache and continuous batching:
1,000 people ask AI", section "How KV cache memory limits concurrency").

Every function is pinned by ``tests/test_oracle_pins.py`` against values and
identities the pages and mathematics fix, not against itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lib = None
_lock = threading.Lock()

_DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float64: 3}


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libpkv_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i, i64, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.pkv_oracle_kv_append.argtypes = [p, p, p, p, p, i64, i64, i, i, i, i]
            lib.pkv_oracle_decode.argtypes = [p, p, p, p, p, p, i, i, i64, i, i, i, i, d, i, p, i]
            lib.pkv_oracle_prefill.argtypes = [p, p, p, p, p, i, i, i, i64, i, i, i, i, d, i, p, i]
            lib.pkv_oracle_causal_attention.argtypes = [p, p, p, p, i, i, i, i, d, i]
            for f in ("pkv_oracle_kv_append", "pkv_oracle_decode", "pkv_oracle_prefill",
                      "pkv_oracle_causal_attention", "pkv_oracle_num_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (set OMP_NUM_THREADS, or set_threads)."""
    return int(_load().pkv_oracle_num_threads())


def set_threads(n: int) -> None:
    """Run later oracle calls on n threads (timing only; results do not change)."""
    lib = _load()
    lib.pkv_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.pkv_oracle_set_threads.restype = None
    lib.pkv_oracle_set_threads(int(n))


def _cpu(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes CPU tensors")
    return t.contiguous()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise RuntimeError(f"oracle {what} failed with status {status}")


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """Bytes of cache one token costs: key and value, per layer, per KV head,
    at the head dimension, at the storage precision."""
    return 2 * layers * kv_heads * head_dim * dtype_bytes


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping) -> None:
    """Scatter k_new/v_new [T, Hkv, D] into pools [NB, Hkv, bs, D] in place,
    byte for byte, at ``slot_mapping`` [T] (int64; negative = skip)."""
    k_new, v_new, slot_mapping = _cpu(k_new), _cpu(v_new), _cpu(slot_mapping)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("pools must be contiguous")
    nb, hkv, bs, d = k_cache.shape
    assert slot_mapping.dtype == torch.int64 and k_new.dtype == k_cache.dtype
    st = _load().pkv_oracle_kv_append(
        k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slot_mapping.data_ptr(), k_new.shape[0], nb, hkv, d, bs, k_new.element_size())
    _check(st, "kv_append")


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale, pairs=None):
    """fp64 decode attention.  q [B, Hq, D]; pools [NB, Hkv, bs, D];
    block_table [B, max_blocks] int32; seq_lens [B] int32 (after the append).
    Returns [B, Hq, D] float64, or [n, D] for ``pairs`` = [(seq, head), ...]."""
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    block_table, seq_lens = _cpu(block_table).to(torch.int32), _cpu(seq_lens).to(torch.int32)
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    if pairs is not None:
        pr = torch.as_tensor(pairs, dtype=torch.int32).reshape(-1, 2).contiguous()
        out = torch.empty(pr.shape[0], d, dtype=torch.float64)
        pp, npairs = pr.data_ptr(), pr.shape[0]
    else:
        out = torch.empty(b, hq, d, dtype=torch.float64)
        pr, pp, npairs = None, None, 0
    st = _load().pkv_oracle_decode(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_table.data_ptr(), seq_lens.data_ptr(), b, block_table.shape[1], nb, hq, hkv, d,
        bs, float(scale), _DTYPE_CODE[q.dtype], pp, npairs)
    _check(st, "decode")
    return out


def chunked_prefill(q, k_cache, v_cache, block_table_row, prior_len, scale, rows=None):
    """fp64 chunked-prefill attention of one sequence.  q [C, Hq, D]; row i sits
    at absolute position prior_len + i and sees keys 0..prior_len+i, read
    through ``block_table_row`` [max_blocks] int32.  Returns [C, Hq, D] float64,
    or [n, D] for ``rows`` = [(row, head), ...]."""
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_table_row).to(torch.int32)
    c, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    if rows is not None:
        pr = torch.as_tensor(rows, dtype=torch.int32).reshape(-1, 2).contiguous()
        out = torch.empty(pr.shape[0], d, dtype=torch.float64)
        pp, n = pr.data_ptr(), pr.shape[0]
    else:
        out = torch.empty(c, hq, d, dtype=torch.float64)
        pr, pp, n = None, None, 0
    st = _load().pkv_oracle_prefill(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), bt.data_ptr(),
        bt.shape[0], int(prior_len), c, nb, hq, hkv, d, bs, float(scale),
        _DTYPE_CODE[q.dtype], pp, n)
    _check(st, "prefill")
    return out


def causal_attention(q, k, v, scale):
    """Recompute path: full causal attention over one contiguous sequence.
    q [T, Hq, D]; k, v [T, Hkv, D]; returns [T, Hq, D] float64."""
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    t, hq, d = q.shape
    hkv = k.shape[1]
    out = torch.empty(t, hq, d, dtype=torch.float64)
    st = _load().pkv_oracle_causal_attention(
        out.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), t, hq, hkv, d,
        float(scale), _DTYPE_CODE[q.dtype])
    _check(st, "causal_attention")
    return out
