"""The C ABI without a GPU: the library builds/loads, exports every function
include/pagedkv.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a machine with no GPU)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="needs nvcc to build the library")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_104_gb300 import binding, build
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("pkv_kv_append", "pkv_paged_decode_attention", "pkv_chunked_prefill_attention"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    nm = shutil.which("nm")
    for name in declared_functions():
        assert hasattr(lib, name), name  # dlsym
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", lib._name], capture_output=True,
                             text=True).stdout
        for name in declared_functions():
            assert re.search(rf"\bT {name}$", out, re.M), name


def test_binding_names_match_header(lib):
    from paged_kv_cache_104_gb300 import binding
    assert set(binding.EXPORTS) == set(declared_functions())
    for short in ("kv_append", "paged_decode_attention", "chunked_prefill_attention",
                  "decode_workspace_bytes", "get_device_error", "status_str", "abi_version"):
        assert callable(getattr(binding, short))


def test_host_only_functions(lib):
    from paged_kv_cache_104_gb300 import binding
    assert binding.abi_version() == 2
    assert binding.status_str(0) == "ok"
    assert binding.status_str(5) == "unsupported shape"
    # one split of 512 tokens needs no workspace; more need (D + 2) floats per
    # partial slot (ceil(L / 512) + 1 slots per row) and one int per row
    assert binding.decode_workspace_bytes(64, 32, 128, 512) == 0
    n = binding.decode_workspace_bytes(64, 32, 128, 2301)
    rows = 64 * 32 * 6
    base = rows * 130 * 4 + 64 * 32 * 4
    assert n >= base and n < base + 768


def _nullp():
    return ctypes.c_void_p(0)


def _fake(addr=0x1000):
    return ctypes.c_void_p(addr)


def test_append_rejects_bad_arguments_on_host(lib):
    f = lib.pkv_kv_append
    P = _fake()
    assert f(P, P, P, P, P, 4, 32, 2, 16, 16, 7, None) == 2          # dtype
    assert f(P, P, P, P, P, -1, 32, 2, 16, 16, 0, None) == 1         # negative tokens
    assert f(P, P, P, P, P, 4, 32, 2, 16, 8, 0, None) == 5           # block size 8
    assert f(P, P, P, P, P, 4, 32, 2, 3, 16, 0, None) == 5           # 12-byte rows
    assert f(_nullp(), P, P, P, P, 4, 32, 2, 16, 16, 0, None) == 1   # null
    assert f(_fake(0x1004), P, P, P, P, 4, 32, 2, 16, 16, 0, None) == 1  # misaligned
    assert f(_nullp(), _nullp(), _nullp(), _nullp(), _nullp(), 0, 32, 2, 16, 16, 0, None) == 0


def test_decode_rejects_bad_arguments_on_host(lib):
    f = lib.pkv_paged_decode_attention
    P = _fake()

    def call(**kw):
        a = dict(out=P, q=P, k=P, v=P, bt=P, sl=P, B=4, mb=4, msl=64, nb=32, hq=4, hkv=2, d=16,
                 bs=16, scale=0.25, ws=_nullp(), wsb=0, dt=0)
        a.update(kw)
        return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["sl"], a["B"], a["mb"], a["msl"],
                 a["nb"], a["hq"], a["hkv"], a["d"], a["bs"], a["scale"], a["ws"], a["wsb"],
                 a["dt"], None)
    assert call(dt=9) == 2
    assert call(hq=6, hkv=4) == 1                 # not a whole group
    assert call(hq=48, hkv=3) == 5                # group 16 not compiled
    assert call(d=64) == 5                        # fp32 head_dim 64 not compiled
    assert call(dt=1, d=16) == 5                  # bf16 head_dim 16 not compiled
    assert call(bs=32) == 5
    assert call(msl=65) == 1                      # beyond max_blocks * block_size
    assert call(B=9000) == 3                      # too many sequences
    assert call(scale=float("nan")) == 1
    assert call(q=_nullp()) == 1
    assert call(out=_fake(0x1008)) == 1
    assert call(B=0) == 0                          # empty batch: no-op
    # two splits need a workspace
    assert call(mb=64, msl=1000, wsb=0) == 3
    assert call(mb=64, msl=1000, wsb=1 << 20, ws=_nullp()) == 1


def test_prefill_rejects_bad_arguments_on_host(lib):
    f = lib.pkv_chunked_prefill_attention
    P = _fake()

    def call(**kw):
        a = dict(out=P, q=P, k=P, v=P, bt=P, mb=8, prior=64, chunk=64, nb=32, hq=32, hkv=8, d=128,
                 bs=16, scale=0.1, dt=1)
        a.update(kw)
        return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["prior"], a["chunk"],
                 a["nb"], a["hq"], a["hkv"], a["d"], a["bs"], a["scale"], a["dt"], None)
    assert call(chunk=0) == 0
    assert call(prior=-1) == 1
    assert call(prior=100) == 1                   # 164 tokens > 8 blocks * 16
    assert call(dt=3) == 2
    assert call(bt=_nullp()) == 1
    assert call(d=96) == 5


def test_span_buffer_setter_on_host(lib):
    """pkv_set_span_buffer takes an 8-byte aligned pointer or NULL; it only
    stores it (no CUDA call), so this runs without a GPU."""
    import ctypes
    assert lib.pkv_set_span_buffer(ctypes.c_void_p(0x1003)) == 1
    assert lib.pkv_set_span_buffer(ctypes.c_void_p(0x1000)) == 0
    assert lib.pkv_set_span_buffer(None) == 0
