"""Plant one plausible mistake at a time in a copy of the oracle's C source,
compile it on the CPU, and require that at least one pin rejects it.

This shows the pins are sharp enough: a dropped term, a wrong index, a
transposed layout or a wrong sign in the oracle would not go unnoticed.
"""
import importlib.util
import os
import shutil
import subprocess

import pytest

import oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

MUTANTS = {
    "gqa_mapping_modulo": ("h / group", "h % num_kv_heads"),
    "scale_dropped": ("w[j] = scale * s;", "w[j] = s;"),
    "exp_sign_flipped": ("w[j] = exp(w[j] - m);", "w[j] = exp(m - w[j]);"),
    "normalisation_dropped": ("out[d] /= z;", "out[d] /= 1.0;"),
    "pool_layout_transposed": (
        "(((int64_t)blk * num_kv_heads + g) * block_size + p % block_size)",
        "(((int64_t)blk * block_size + p % block_size) * num_kv_heads + g)"),
    "block_row_wrong": ("bt_row[p / block_size]", "bt_row[p % block_size]"),
    "decode_misses_own_key": ("int64_t n = seq_lens[b];", "int64_t n = seq_lens[b] - 1 + (seq_lens[b] == 1);"),
    "prefill_causal_off_by_one": ("int64_t n = (int64_t)prior_len + i + 1;",
                                  "int64_t n = (int64_t)prior_len + i + (i == 0);"),
    "append_value_into_key_pool": ("memcpy((char *)v_cache + dst, (const char *)v_new + src",
                                   "memcpy((char *)v_cache + dst, (const char *)k_new + src"),
    "append_wrong_head_offset": ("int64_t src = ((t * num_kv_heads) + h) * row_bytes;",
                                 "int64_t src = ((t * num_kv_heads)) * row_bytes;"),
    "score_uses_value": ("s += q[d] * kc[j * head_dim + d];", "s += q[d] * vc[j * head_dim + d];"),
    "bf16_widening_wrong_shift": ("<< 16;", "<< 15;"),
}


def _build_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    d = tmp_path / name
    d.mkdir()
    src = d / "pkv_oracle.c"
    src.write_text(text.replace(old, new))
    lib = d / "libpkv_oracle.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib),
                    str(src), "-lm"], check=True)
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}",
                                                  os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC, mod._BUILD_DIR, mod._LIB_PATH = str(src), str(d), str(lib)
    return mod


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    mod = _build_mutant(name, tmp_path)
    failed = []
    for check in P.ALL_CHECKS:
        try:
            check(mod)
        except (AssertionError, RuntimeError) as e:  # RuntimeError: oracle status
            failed.append(check.__name__)
    assert failed, f"no pin caught mutant {name}"
