"""Prefix-caching oracle: chained block identifiers and prefix matching.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Plain Python, written
independently of the library's C++ (paged_kv_cache_104_gb300/csrc/prefix_cache.cpp).

Rules from "The KV cache and prefix caching", section "A prefix already in
the cache can skip its prefill":
  * the prompt is hashed block by block (16 tokens per block);
  * each block's identifier covers its tokens and the identifier of the block
    before it, so equal identifiers mean equal prefixes up to that block and a
    match is a contiguous prefix starting at position 0;
  * a hit is counted in whole blocks; the last partial block is recomputed.
Readings where the page is silent:
  * the hash is 64-bit FNV-1a (Fowler/Noll/Vo), fed the previous identifier as
    8 little-endian bytes then each token id as 4 little-endian bytes; the
    first block's previous identifier is 0;
  * at least the prompt's last token is always recomputed (it must produce the
    first output token), so a fully cached whole-block prompt reuses all but
    its last block.
"""
from __future__ import annotations

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    h = FNV_OFFSET
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK
    return h


def block_ids(tokens, block_size: int = 16, parent: int = 0) -> list:
    """Identifiers of the full blocks of ``tokens``, each chained to the one before."""
    out = []
    prev = parent
    for b in range(len(tokens) // block_size):
        data = prev.to_bytes(8, "little")
        for t in tokens[b * block_size:(b + 1) * block_size]:
            data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
        prev = fnv1a64(data)
        out.append(prev)
    return out


class PrefixIndex:
    """identifier -> physical block; the first block recorded for an identifier stays."""

    def __init__(self):
        self.table = {}

    def insert(self, ids, blocks):
        for i, b in zip(ids, blocks):
            self.table.setdefault(i, b)

    def match(self, ids):
        blocks = []
        for i in ids:
            if i not in self.table:
                break
            blocks.append(self.table[i])
        return len(blocks), blocks

    def plan(self, tokens, block_size: int = 16):
        """Reusable prompt tokens (whole blocks, at most len-1) and their blocks."""
        ids = block_ids(tokens, block_size)
        usable = (len(tokens) - 1) // block_size
        m, blocks = self.match(ids[:usable])
        return m * block_size, blocks, ids
