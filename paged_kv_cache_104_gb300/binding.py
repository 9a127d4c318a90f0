"""Thin Python binding of libpagedkv.so (argument marshalling only).

Every function takes torch CUDA tensors, passes their device pointers, sizes
and the current CUDA stream to the C ABI of the same name (``include/pagedkv.h``)
and raises ``PagedKVError`` on a non-zero status.  No step of the computation
runs here: if the library is missing the import of a function fails loudly
instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")
_lib = None
_lock = threading.Lock()

PKV_F32, PKV_BF16 = 0, 1
DEVERR = {0: "none", 1: "slot out of range", 2: "block id out of range",
          3: "sequence length out of range", 4: "internal wait timed out",
          5: "shared-memory layout check failed"}
EXPORTS = ("pkv_kv_append", "pkv_decode_workspace_bytes", "pkv_paged_decode_attention",
           "pkv_paged_decode_attention_append", "pkv_paged_decode_attention_noalloc", "pkv_chunked_prefill_attention",
           "pkv_decode_prefill_attention",
           "pkv_get_device_error", "pkv_status_str", "pkv_abi_version",
           "pkv_kv_append_fp8", "pkv_paged_decode_attention_fp8",
           "pkv_latent_append", "pkv_mla_workspace_bytes", "pkv_mla_decode_attention",
           "pkv_mla_decode_attention_append",
           "pkv_fnv1a64", "pkv_prefix_hash_blocks", "pkv_prefix_cache_create",
           "pkv_prefix_cache_destroy", "pkv_prefix_cache_size", "pkv_prefix_cache_insert",
           "pkv_prefix_cache_evict", "pkv_prefix_cache_match", "pkv_prefix_plan",
           "pkv_l2_flush", "pkv_set_span_buffer")
NOALLOC_SCRATCH_BYTES = 32 << 20  # PKV_NOALLOC_SCRATCH_BYTES


class DecodePrefillArgs(ctypes.Structure):
    """pkv_decode_prefill_args (field order and types as in pagedkv.h)."""
    _fields_ = [("decode_out", ctypes.c_void_p), ("decode_q", ctypes.c_void_p),
                ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("max_seq_len", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("prefill_out", ctypes.c_void_p),
                ("prefill_q", ctypes.c_void_p), ("prefill_block_table", ctypes.c_void_p),
                ("prefill_max_blocks", ctypes.c_int), ("prior_len", ctypes.c_int),
                ("chunk_len", ctypes.c_int), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int), ("prefill_sms", ctypes.c_int),
                ("chunk_k_new", ctypes.c_void_p), ("chunk_v_new", ctypes.c_void_p),
                ("chunk_slot_mapping", ctypes.c_void_p)]


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def open_library(path: str):
    """Load a build of the library at ``path`` and declare its argument types."""
    lib = ctypes.CDLL(path)
    p, i, i64, f, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                        ctypes.c_size_t)
    lib.pkv_kv_append.argtypes = [p, p, p, p, p, i64, i64, i, i, i, i, p]
    lib.pkv_decode_workspace_bytes.argtypes = [i, i, i, i]
    lib.pkv_decode_workspace_bytes.restype = sz
    lib.pkv_paged_decode_attention.argtypes = [p, p, p, p, p, p, i, i, i, i64, i, i, i, i, f,
                                               p, sz, i, p]
    lib.pkv_chunked_prefill_attention.argtypes = [p, p, p, p, p, i, i, i, i64, i, i, i, i, f,
                                                  i, p]
    lib.pkv_paged_decode_attention_noalloc.argtypes = [p, p, p, p, p, p, i, i, i, i64, i, i,
                                                       i, i, f, i, p]
    lib.pkv_paged_decode_attention_append.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i64, i,
                                                      i, i, i, f, p, sz, i, p]
    lib.pkv_decode_prefill_attention.argtypes = [ctypes.POINTER(DecodePrefillArgs), p]
    lib.pkv_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), i]
    lib.pkv_l2_flush.argtypes = [p, sz, p, p]
    lib.pkv_l2_flush.restype = ctypes.c_int
    lib.pkv_set_span_buffer.argtypes = [p]
    lib.pkv_set_span_buffer.restype = ctypes.c_int
    lib.pkv_status_str.argtypes = [i]
    lib.pkv_status_str.restype = ctypes.c_char_p
    lib.pkv_kv_append_fp8.argtypes = [p, p, p, p, p, p, p, i64, i64, i, i, i, p]
    lib.pkv_kv_append_fp8.restype = ctypes.c_int
    lib.pkv_paged_decode_attention_fp8.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i64, i, i,
                                                   i, i, f, p, sz, p]
    lib.pkv_paged_decode_attention_fp8.restype = ctypes.c_int
    lib.pkv_latent_append.argtypes = [p, p, p, i64, i64, i, i, p]
    lib.pkv_latent_append.restype = ctypes.c_int
    lib.pkv_mla_workspace_bytes.argtypes = [i, i, i, i]
    lib.pkv_mla_workspace_bytes.restype = sz
    lib.pkv_mla_decode_attention.argtypes = [p, p, p, p, p, p, p, i, i, i, i64, i, i, i, i, f,
                                             p, sz, p]
    lib.pkv_mla_decode_attention.restype = ctypes.c_int
    lib.pkv_mla_decode_attention_append.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i64, i, i, i,
                                                    i, f, p, sz, p]
    lib.pkv_mla_decode_attention_append.restype = ctypes.c_int
    u64p = ctypes.POINTER(ctypes.c_uint64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.pkv_fnv1a64.argtypes = [p, sz]
    lib.pkv_fnv1a64.restype = ctypes.c_uint64
    lib.pkv_prefix_hash_blocks.argtypes = [i32p, i64, i, ctypes.c_uint64, u64p]
    lib.pkv_prefix_hash_blocks.restype = i64
    lib.pkv_prefix_cache_create.argtypes = []
    lib.pkv_prefix_cache_create.restype = p
    lib.pkv_prefix_cache_destroy.argtypes = [p]
    lib.pkv_prefix_cache_destroy.restype = None
    lib.pkv_prefix_cache_size.argtypes = [p]
    lib.pkv_prefix_cache_size.restype = i64
    lib.pkv_prefix_cache_insert.argtypes = [p, u64p, i32p, i64]
    lib.pkv_prefix_cache_insert.restype = ctypes.c_int
    lib.pkv_prefix_cache_evict.argtypes = [p, u64p, i64]
    lib.pkv_prefix_cache_evict.restype = ctypes.c_int
    lib.pkv_prefix_cache_match.argtypes = [p, u64p, i64, i32p]
    lib.pkv_prefix_cache_match.restype = i64
    lib.pkv_prefix_plan.argtypes = [p, i32p, i64, i, i32p, u64p]
    lib.pkv_prefix_plan.restype = i64
    for name in ("pkv_kv_append", "pkv_paged_decode_attention",
                 "pkv_paged_decode_attention_noalloc", "pkv_paged_decode_attention_append",
                 "pkv_chunked_prefill_attention", "pkv_decode_prefill_attention",
                 "pkv_get_device_error", "pkv_abi_version"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def load():
    """Load the shared library (built by ``paged_kv_cache_104_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m paged_kv_cache_104_gb300.build`")
        _lib = open_library(LIB_PATH)
        return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    if t.dtype == torch.float32:
        return PKV_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise PagedKVError(fn, status, load().pkv_status_str(status).decode())


# debug mode: host-side checks of the index arrays before each call
_debug = os.environ.get("PKV_DEBUG", "") not in ("", "0")


def set_debug(flag: bool) -> None:
    """Turn the host-side index checks (``validate.py``) on or off."""
    global _debug
    _debug = bool(flag)


def _validate(fn: str, check: str, *args, **kw) -> None:
    """In debug mode, run validate.<check>(*args, **kw) before the call."""
    if not _debug:
        return
    from . import validate as V
    try:
        getattr(V, check)(*args, **kw)
    except V.ValidationError as e:
        raise PagedKVError(fn, V.PKV_EINVAL, str(e)) from None


def status_str(status: int) -> str:
    return load().pkv_status_str(status).decode()


def abi_version() -> int:
    return int(load().pkv_abi_version())


def l2_flush(buf, sink, stream=None) -> None:
    """Measurement helper: read the device buffer ``buf`` (several times the
    L2's size) so the next launch finds none of its inputs in L2; ``sink`` is
    a device int32 the kernel may write."""
    st = load().pkv_l2_flush(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                             _stream(stream))
    _check("pkv_l2_flush", st)


def set_span_buffer(buf=None) -> None:
    """Record the side-by-side call's half spans into buf (int64 [4] on the
    device, initialised by the caller); None turns it off."""
    _check("pkv_set_span_buffer", load().pkv_set_span_buffer(_ptr(buf)))


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """k_new, v_new [T, Hkv, D]; pools [NB, Hkv, bs, D]; slot_mapping [T] int64."""
    nb, hkv, bs, d = k_cache.shape
    _validate("pkv_kv_append", "check_slots", slot_mapping, nb, bs)
    st = load().pkv_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                              _ptr(slot_mapping), int(slot_mapping.shape[0]), nb, hkv, d, bs,
                              _dtype_code(k_cache), _stream(stream))
    _check("pkv_kv_append", st)


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_seq_len: int) -> int:
    return int(load().pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len))


def decode_workspace(num_seqs, num_q_heads, head_dim, max_seq_len, device="cuda"):
    """Allocate (through torch) the workspace paged_decode_attention needs."""
    n = decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def paged_decode_attention(out, q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int,
                           scale: float, workspace=None, stream=None) -> None:
    """out, q [B, Hq, D]; pools [NB, Hkv, bs, D]; block_table [B, max_blocks]
    int32; seq_lens [B] int32 (after the append); max_seq_len >= max(seq_lens)."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _validate("pkv_paged_decode_attention", "check_decode", block_table, seq_lens,
              max_seq_len, nb, bs)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pkv_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        b, int(block_table.shape[1]), int(max_seq_len), nb, hq, hkv, d, bs, float(scale),
        _ptr(workspace), ws_bytes, _dtype_code(q), _stream(stream))
    _check("pkv_paged_decode_attention", st)


def paged_decode_attention_append(out, q, k_new, v_new, k_cache, v_cache, block_table, seq_lens,
                                  max_seq_len: int, scale: float, workspace=None,
                                  stream=None) -> None:
    """Append each sequence's new key/value (k_new, v_new [B, Hkv, D]) at
    position seq_lens[b] - 1 and attend, in one launch."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _validate("pkv_paged_decode_attention_append", "check_decode", block_table,
              seq_lens, max_seq_len, nb, bs, appends=True)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pkv_paged_decode_attention_append(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), _ptr(seq_lens), b, int(block_table.shape[1]), int(max_seq_len), nb, hq,
        hkv, d, bs, float(scale), _ptr(workspace), ws_bytes, _dtype_code(q), _stream(stream))
    _check("pkv_paged_decode_attention_append", st)


def kv_append_fp8(k_new, v_new, k_cache, v_cache, k_scale, v_scale, slot_mapping,
                  stream=None) -> None:
    """bf16 k_new, v_new [T, Hkv, D] -> E4M3 codes of x / scale[h] in uint8
    pools [NB, Hkv, bs, D]; k_scale, v_scale float32 [Hkv] on the device."""
    nb, hkv, bs, d = k_cache.shape
    _validate("pkv_kv_append_fp8", "check_slots", slot_mapping, nb, bs)
    st = load().pkv_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(k_scale), _ptr(v_scale), _ptr(slot_mapping),
                                  int(slot_mapping.shape[0]), nb, hkv, d, bs, _stream(stream))
    _check("pkv_kv_append_fp8", st)


def paged_decode_attention_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                               max_seq_len: int, scale: float, workspace=None, stream=None) -> None:
    """Decode over uint8 E4M3 pools; q/out bf16 [B, Hq, D]."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _validate("pkv_paged_decode_attention_fp8", "check_decode", block_table, seq_lens,
              max_seq_len, nb, bs)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().pkv_paged_decode_attention_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_table), _ptr(seq_lens), b, int(block_table.shape[1]), int(max_seq_len), nb, hq,
        hkv, d, bs, float(scale), _ptr(workspace), ws_bytes, _stream(stream))
    _check("pkv_paged_decode_attention_fp8", st)


def latent_append(c_new, c_cache, slot_mapping, stream=None) -> None:
    """bf16 c_new [T, r] -> latent pool [NB, bs, r] at slot_mapping (int64)."""
    nb, bs, r = c_cache.shape
    _validate("pkv_latent_append", "check_slots", slot_mapping, nb, bs)
    st = load().pkv_latent_append(_ptr(c_new), _ptr(c_cache), _ptr(slot_mapping),
                                  int(slot_mapping.shape[0]), nb, r, bs, _stream(stream))
    _check("pkv_latent_append", st)


def mla_workspace(num_seqs: int, num_q_heads: int, rank: int, max_seq_len: int, device=None):
    n = int(load().pkv_mla_workspace_bytes(num_seqs, num_q_heads, rank, max_seq_len))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def mla_decode_attention(out, q, w_k, w_v, c_cache, block_table, seq_lens, max_seq_len: int,
                         scale: float, workspace=None, stream=None, c_new=None) -> None:
    """Decode over the latent pool [NB, bs, r]; q/out bf16 [B, Hq, D];
    w_k, w_v bf16 [Hq, D, r].  With c_new [B, r] each sequence's new latent is
    first placed at position seq_lens[b] - 1 (the same call)."""
    b, hq, d = q.shape
    nb, bs, r = c_cache.shape
    _validate("pkv_mla_decode_attention", "check_decode", block_table, seq_lens,
              max_seq_len, nb, bs, appends=c_new is not None)
    if workspace is None:
        workspace = mla_workspace(b, hq, r, max_seq_len, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if c_new is not None:
        st = load().pkv_mla_decode_attention_append(
            _ptr(out), _ptr(q), _ptr(c_new), _ptr(w_k), _ptr(w_v), _ptr(c_cache),
            _ptr(block_table), _ptr(seq_lens), b, int(block_table.shape[1]), int(max_seq_len), nb,
            hq, d, r, bs, float(scale), _ptr(workspace), ws_bytes, _stream(stream))
        _check("pkv_mla_decode_attention_append", st)
        return
    st = load().pkv_mla_decode_attention(
        _ptr(out), _ptr(q), _ptr(w_k), _ptr(w_v), _ptr(c_cache), _ptr(block_table),
        _ptr(seq_lens), b, int(block_table.shape[1]), int(max_seq_len), nb, hq, d, r, bs,
        float(scale), _ptr(workspace), ws_bytes, _stream(stream))
    _check("pkv_mla_decode_attention", st)


def paged_decode_attention_noalloc(out, q, k_cache, v_cache, block_table, seq_lens,
                                   max_seq_len: int, scale: float, stream=None) -> None:
    """paged_decode_attention without a workspace argument: the split partials
    go to a scratch array inside the library (NOALLOC_SCRATCH_BYTES, shared by
    every call; calls that overlap on the GPU race).  For callers that may not
    allocate device memory."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _validate("pkv_paged_decode_attention_noalloc", "check_decode", block_table,
              seq_lens, max_seq_len, nb, bs)
    st = load().pkv_paged_decode_attention_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        b, int(block_table.shape[1]), int(max_seq_len), nb, hq, hkv, d, bs, float(scale),
        _dtype_code(q), _stream(stream))
    _check("pkv_paged_decode_attention_noalloc", st)


def chunked_prefill_attention(out, q, k_cache, v_cache, block_table_row, prior_len: int,
                              scale: float, stream=None) -> None:
    """out, q [C, Hq, D]; block_table_row [max_blocks] int32; the chunk sits at
    positions prior_len .. prior_len+C-1 and its K/V are already appended."""
    c, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _validate("pkv_chunked_prefill_attention", "check_prefill", block_table_row,
              prior_len, c, nb, bs)
    st = load().pkv_chunked_prefill_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table_row),
        int(block_table_row.shape[0]), int(prior_len), c, nb, hq, hkv, d, bs, float(scale),
        _dtype_code(q), _stream(stream))
    _check("pkv_chunked_prefill_attention", st)


def decode_prefill_attention(dec_out, dec_q, k_new, v_new, k_cache, v_cache, block_table, seq_lens,
                             max_seq_len: int, pre_out, pre_q, pre_block_table_row, prior_len: int,
                             scale: float, workspace=None, prefill_sms: int = 0,
                             stream=None, chunk_k_new=None, chunk_v_new=None,
                             chunk_slots=None) -> None:
    """One layer's decode (as paged_decode_attention_append) and one chunk's
    prefill (as chunked_prefill_attention) side by side on disjoint SMs:
    prefill_sms SMs for the prefill (0: a quarter of the GPU).  With
    chunk_k_new / chunk_v_new [chunk, Hkv, D] and chunk_slots (int64 [chunk])
    the call first appends the chunk's own keys and values (as kv_append)."""
    b, hq, d = dec_q.shape
    nb, hkv, bs, _ = k_cache.shape
    _validate("pkv_decode_prefill_attention", "check_decode", block_table, seq_lens,
              max_seq_len, nb, bs, appends=True)
    _validate("pkv_decode_prefill_attention", "check_prefill", pre_block_table_row,
              prior_len, int(pre_q.shape[0]), nb, bs)
    if chunk_slots is not None:
        _validate("pkv_decode_prefill_attention", "check_slots", chunk_slots, nb, bs)
    a = DecodePrefillArgs()
    a.decode_out, a.decode_q = _ptr(dec_out), _ptr(dec_q)
    a.k_new, a.v_new = _ptr(k_new), _ptr(v_new)
    a.block_table, a.seq_lens = _ptr(block_table), _ptr(seq_lens)
    a.num_seqs, a.max_blocks_per_seq, a.max_seq_len = b, int(block_table.shape[1]), int(max_seq_len)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.prefill_out, a.prefill_q = _ptr(pre_out), _ptr(pre_q)
    a.prefill_block_table = _ptr(pre_block_table_row)
    a.prefill_max_blocks = int(pre_block_table_row.shape[0])
    a.prior_len, a.chunk_len = int(prior_len), int(pre_q.shape[0])
    a.k_cache, a.v_cache, a.num_blocks = _ptr(k_cache), _ptr(v_cache), nb
    a.num_q_heads, a.num_kv_heads, a.head_dim, a.block_size = hq, hkv, d, bs
    a.scale, a.dtype, a.prefill_sms = float(scale), _dtype_code(dec_q), int(prefill_sms)
    a.chunk_k_new, a.chunk_v_new = _ptr(chunk_k_new), _ptr(chunk_v_new)
    a.chunk_slot_mapping = _ptr(chunk_slots)
    st = load().pkv_decode_prefill_attention(ctypes.byref(a), _stream(stream))
    _check("pkv_decode_prefill_attention", st)


def get_device_error(clear: bool = True) -> int:
    """Device error word of the current device (0 = none); synchronises."""
    code = ctypes.c_int(0)
    _check("pkv_get_device_error", load().pkv_get_device_error(ctypes.byref(code), int(clear)))
    return code.value


# ----------------------------------------------------------------- prefix cache
def fnv1a64(data: bytes) -> int:
    return int(load().pkv_fnv1a64(ctypes.c_char_p(bytes(data)), len(data)))


def _i32(a):
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _u64(a):
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.uint64))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))


def prefix_hash_blocks(tokens, block_size: int = 16, parent: int = 0):
    """Chained FNV-1a identifiers of the full blocks of a token list."""
    import numpy as np
    toks, tp = _i32(tokens)
    out = np.zeros(max(len(toks) // block_size, 1), dtype=np.uint64)
    n = load().pkv_prefix_hash_blocks(tp, len(toks), block_size, ctypes.c_uint64(parent),
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
    if n < 0:
        raise PagedKVError("pkv_prefix_hash_blocks", 1, "invalid argument")
    return [int(x) for x in out[:n]]


class PrefixCache:
    """Host-side index from chained block identifiers to physical blocks."""

    def __init__(self):
        self._h = load().pkv_prefix_cache_create()
        if not self._h:
            raise MemoryError("pkv_prefix_cache_create")

    def __del__(self):
        if getattr(self, "_h", None):
            load().pkv_prefix_cache_destroy(self._h)
            self._h = None

    def __len__(self):
        return int(load().pkv_prefix_cache_size(self._h))

    def insert(self, hashes, block_ids):
        h, hp = _u64(hashes)
        b, bp = _i32(block_ids)
        assert len(h) == len(b)
        _check("pkv_prefix_cache_insert", load().pkv_prefix_cache_insert(self._h, hp, bp, len(h)))

    def evict(self, hashes):
        h, hp = _u64(hashes)
        _check("pkv_prefix_cache_evict", load().pkv_prefix_cache_evict(self._h, hp, len(h)))

    def match(self, hashes):
        """(number of leading identifiers cached, their physical blocks)."""
        import numpy as np
        h, hp = _u64(hashes)
        out = np.zeros(max(len(h), 1), dtype=np.int32)
        m = load().pkv_prefix_cache_match(self._h, hp, len(h),
                                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        return int(m), [int(x) for x in out[:m]]

    def plan(self, tokens, block_size: int = 16):
        """(reusable prompt tokens, reused physical blocks, every full-block identifier)."""
        import numpy as np
        toks, tp = _i32(tokens)
        nb = max(len(toks) // block_size, 1)
        blocks = np.zeros(nb, dtype=np.int32)
        hashes = np.zeros(nb, dtype=np.uint64)
        m = load().pkv_prefix_plan(self._h, tp, len(toks), block_size,
                                   blocks.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                   hashes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
        if m < 0:
            raise PagedKVError("pkv_prefix_plan", 1, "invalid argument")
        nfull = len(toks) // block_size
        return int(m), [int(x) for x in blocks[: m // block_size]], [int(x) for x in hashes[:nfull]]
