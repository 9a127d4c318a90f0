"""Prefix caching: the oracle against published hash vectors and the page's
rules, and the library's host calls against the oracle (CPU only)."""
import json
import os
import random

import pytest

from oracle import prefix as OP

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "prefix_cache.json")))


def _prompt(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 128256) for _ in range(n)]


# ------------------------------------------------------------------ oracle pins
def test_fnv1a_published_vectors():
    for text, hexval in GOLDEN["fnv1a64_vectors"]["cases"]:
        assert OP.fnv1a64(text.encode()) == int(hexval, 16), text


def test_match_must_start_at_position_zero():
    """A prompt differing only at token 3 shares nothing, however long the rest."""
    base = _prompt(1800, 1)
    idx = OP.PrefixIndex()
    ids = OP.block_ids(base)
    idx.insert(ids, list(range(len(ids))))
    other = list(base)
    other[3] += 1
    assert idx.match(OP.block_ids(other)) == (0, [])
    # identical block contents at a different position do not match either
    shifted = _prompt(16, 9) + base[:1784]
    m, _ = idx.match(OP.block_ids(shifted))
    assert m == 0


def test_prefix_matches_in_whole_blocks_and_recomputes_the_partial_one():
    g = GOLDEN["shared_system_prompt"]
    system = _prompt(g["shared_tokens"], 2)
    first = system + _prompt(g["prompt_tokens"] - g["shared_tokens"], 3)
    second = system + _prompt(g["prompt_tokens"] - g["shared_tokens"], 4)
    idx = OP.PrefixIndex()
    ids = OP.block_ids(first, g["block_size"])
    idx.insert(ids, list(range(100, 100 + len(ids))))
    reused, blocks, _ = idx.plan(second, g["block_size"])
    assert reused == g["reused_tokens"]
    assert g["prompt_tokens"] - reused == g["recomputed_tokens"]
    assert blocks == list(range(100, 100 + reused // 16))


def test_fully_cached_prompt_still_computes_its_last_token():
    p = _prompt(64, 5)
    idx = OP.PrefixIndex()
    ids = OP.block_ids(p)
    idx.insert(ids, [7, 8, 9, 10])
    reused, blocks, _ = idx.plan(p)
    assert reused == 48 and blocks == [7, 8, 9]
    reused, _, _ = idx.plan(p + [1])      # one more token: all four blocks reusable
    assert reused == 64


def test_chain_changes_with_any_earlier_token():
    p = _prompt(160, 6)
    ids = OP.block_ids(p)
    for pos in (0, 15, 16, 100, 159):
        q = list(p)
        q[pos] ^= 1
        qi = OP.block_ids(q)
        b = pos // 16
        assert qi[:b] == ids[:b]                          # blocks before the change agree
        assert all(x != y for x, y in zip(qi[b:], ids[b:]))  # every later block differs


# ------------------------------------------------------------------ library vs oracle
@pytest.fixture(scope="module")
def B():
    from paged_kv_cache_104_gb300 import binding, build
    build.build()
    return binding


def test_library_fnv_and_chained_ids_match_oracle(B):
    for text, hexval in GOLDEN["fnv1a64_vectors"]["cases"]:
        assert B.fnv1a64(text.encode()) == int(hexval, 16)
    for n, seed in ((0, 1), (15, 2), (16, 3), (47, 4), (2000, 5)):
        p = _prompt(n, seed)
        assert B.prefix_hash_blocks(p) == OP.block_ids(p)
    assert B.prefix_hash_blocks(_prompt(40, 6), parent=12345) == OP.block_ids(_prompt(40, 6), parent=12345)


def test_library_index_matches_oracle_on_random_traffic(B):
    r = random.Random(7)
    systems = [_prompt(r.randrange(16, 600), 100 + i) for i in range(5)]
    lib, ora = B.PrefixCache(), OP.PrefixIndex()
    next_block = 0
    for step in range(60):
        prompt = list(r.choice(systems)) + _prompt(r.randrange(1, 300), 1000 + step)
        if r.random() < 0.1:
            prompt[r.randrange(len(prompt))] ^= 1
        got = lib.plan(prompt)
        want = ora.plan(prompt)
        assert got == want, step
        reused, blocks, ids = want
        n_new = len(ids) - reused // 16
        new_blocks = list(range(next_block, next_block + n_new))
        next_block += n_new
        lib.insert(ids[reused // 16:], new_blocks)
        ora.insert(ids[reused // 16:], new_blocks)
        assert len(lib) == len(ora.table)
        if step % 20 == 19:  # evict a few
            victims = list(ora.table)[:10]
            lib.evict(victims)
            for v in victims:
                del ora.table[v]
