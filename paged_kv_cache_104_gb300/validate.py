"""Host-side checks of the index arrays a call reads on the device (a debug aid).

The kernels skip out-of-range slots, block ids and lengths and report them in
the device error word; they never trap.  With the binding's debug mode on
(``PKV_DEBUG=1`` or ``binding.set_debug(True)``) these checks run first, on
host copies of the arrays (each copy synchronises), and raise
``PagedKVError`` with ``PKV_EINVAL`` and a message that names the offending
entry.  They read index arrays only and compute nothing of the attention.
"""
from __future__ import annotations

import torch

PKV_EINVAL = 1


class ValidationError(ValueError):
    """A bad index array; the binding re-raises it as PagedKVError."""


def _host(t):
    return t.detach().to("cpu") if t.is_cuda else t.detach()


def check_slots(slot_mapping, num_blocks: int, block_size: int) -> None:
    """Slots (int64 [T]): negative means skip; the others must lie inside the
    pool and be distinct (two tokens writing one row is a caller error)."""
    s = _host(slot_mapping).to(torch.int64)
    live = s[s >= 0]
    bad = live[live >= num_blocks * block_size]
    if bad.numel():
        raise ValidationError(f"slot {int(bad[0])} outside the pool of {num_blocks} blocks "
                              f"x {block_size} rows")
    if live.numel() != torch.unique(live).numel():
        vals, counts = torch.unique(live, return_counts=True)
        raise ValidationError(f"slot {int(vals[counts > 1][0])} appears more than once")


def check_decode(block_table, seq_lens, max_seq_len: int, num_blocks: int, block_size: int,
                 appends: bool = False) -> None:
    """Every length in [1, min(max_seq_len, blocks per row x block_size)];
    every block id a sequence uses inside the pool.  appends: the call also
    writes each sequence's new token at position seq_lens[b] - 1, so those
    rows must be distinct."""
    bt = _host(block_table).to(torch.int64)
    lens = _host(seq_lens).to(torch.int64)
    limit = min(int(max_seq_len), bt.shape[1] * block_size)
    for b, n in enumerate(lens.tolist()):
        if n < 1 or n > limit:
            raise ValidationError(f"seq_lens[{b}] = {n} outside [1, {limit}]")
        used = bt[b, :(n + block_size - 1) // block_size]
        bad = used[(used < 0) | (used >= num_blocks)]
        if bad.numel():
            raise ValidationError(f"block_table[{b}] holds block {int(bad[0])} outside "
                                  f"[0, {num_blocks})")
    if appends and lens.numel():
        pos = lens - 1
        rows = bt[torch.arange(lens.numel()), pos // block_size] * block_size + pos % block_size
        check_slots(rows, num_blocks, block_size)


def check_prefill(block_table_row, prior_len: int, chunk_len: int, num_blocks: int,
                  block_size: int) -> None:
    """The chunk's sequence holds prior_len + chunk_len tokens: every block id
    covering them inside the pool."""
    row = _host(block_table_row).to(torch.int64)
    n = int(prior_len) + int(chunk_len)
    need = (n + block_size - 1) // block_size
    if need > row.numel():
        raise ValidationError(f"{n} tokens need {need} blocks, the row holds {row.numel()}")
    used = row[:need]
    bad = used[(used < 0) | (used >= num_blocks)]
    if bad.numel():
        raise ValidationError(f"prefill block table holds block {int(bad[0])} outside "
                              f"[0, {num_blocks})")
