"""Seeded synthetic workloads for paged decode / chunked prefill.

This module only draws inputs: context lengths, a shuffled physical block
pool with per-sequence block tables, slot numbers for the appended tokens,
and N(0, 1) queries, keys and values.  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

The five shapes follow the pages' worked sizes: a tiny fp32 case; a toy
decode batch at context 64 ("KV cache and continuous batching: 1,000 people
ask AI", section "What our lab measured"); a Llama-3.1-8B-shaped batch at
context 2,300 with 32 query heads, 8 KV heads and head dimension 128 ("The
KV cache and prefix caching", section "What prefill stores and decode
reads"); a ragged continuous batch plus one 2,048-token prefill chunk ("The
KV cache is not your bottleneck", section "The fix that mattered"); and a
long-context batch at 32,000 tokens ("The KV cache and prefix caching",
section "The prompt is paid once, the output is paid every step").

Layout conventions (shared with the C ABI):
  pools        [num_blocks, Hkv, block_size, D]
  block_table  [rows, max_blocks] int32 (unused tail entries hold valid but
               unrelated block ids, so a kernel that wrongly read them would
               give a wrong answer rather than touch memory outside the pool)
  seq_lens     [B] int32, tokens stored after this step's append
  slot_mapping [T] int64 = block * block_size + row, for each appended token
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_seqs: int
    seed: int
    context: tuple = ()                # fixed cached lengths (before the step)
    context_loguniform: tuple = ()     # (lo, hi): floor(exp(U(ln lo, ln hi)))
    prefill_chunk: int = 0             # prompt tokens of the one prefill chunk
    prefill_prior: int = 0             # tokens that chunk's sequence already has
    pool_blocks: int = 0               # explicit pool size (0: needed + spare)
    spare_frac: float = 0.03           # unused blocks added to the pool
    description: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", torch.float32, layers=1, num_q_heads=4, num_kv_heads=2, head_dim=16,
        block_size=16, num_seqs=4, seed=0, context=(5, 17, 33, 64), pool_blocks=32,
        description="fp32, 4 q / 2 kv heads, D 16, cached {5,17,33,64}, pool of 32 blocks"),
    "toy_decode": Workload(
        "toy_decode", torch.bfloat16, layers=1, num_q_heads=32, num_kv_heads=8, head_dim=128,
        block_size=16, num_seqs=16, seed=1, context=(64,) * 16,
        description="bf16, 32/8/128, 16 sequences at context 64"),
    "llama8b_decode": Workload(
        "llama8b_decode", torch.bfloat16, layers=32, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, num_seqs=64, seed=2, context=(2300,) * 64,
        description="bf16, 32 layers, 32/8/128, 64 sequences at context 2,300"),
    "ragged_prefill": Workload(
        "ragged_prefill", torch.bfloat16, layers=32, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, num_seqs=128, seed=3, context_loguniform=(128, 32768),
        prefill_chunk=2048, prefill_prior=4096,
        description="bf16, 32 layers, 32/8/128, 128 decode sequences at log-uniform "
                    "context in [128, 32768] plus a 2,048-token chunk over 4,096 cached tokens"),
    "long_context": Workload(
        "long_context", torch.bfloat16, layers=32, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, num_seqs=8, seed=4, context=(32000,) * 8,
        description="bf16, 32 layers, 32/8/128, 8 sequences at context 32,000"),
}


def context_lens(w: Workload) -> torch.Tensor:
    """Cached tokens per decode sequence before the step (int64 [B])."""
    if w.context:
        assert len(w.context) == w.num_seqs
        return torch.tensor(w.context, dtype=torch.int64)
    lo, hi = w.context_loguniform
    g = torch.Generator().manual_seed(1000 + w.seed)
    u = torch.rand(w.num_seqs, generator=g, dtype=torch.float64)
    lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return lens.clamp(lo, hi).to(torch.int64)


@dataclass
class Layout:
    """Block pool, block tables and slots for one step of one workload."""
    seq_lens: torch.Tensor        # [B] int32, decode sequences after the append
    block_table: torch.Tensor     # [B (+1 prefill row), max_blocks] int32
    num_blocks: int
    slot_mapping: torch.Tensor    # [T] int64, decode tokens then prefill tokens
    num_decode_tokens: int
    prefill_row: int              # row of block_table of the prefill sequence, or -1
    used_blocks: int

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def decode_block_table(self) -> torch.Tensor:
        n = self.seq_lens.shape[0]
        return self.block_table[:n]


def make_layout(w: Workload, seq_lens_after=None, prefill=None, seed_offset: int = 0) -> Layout:
    """Deal a uniformly shuffled physical pool out to the sequences.

    ``seq_lens_after`` overrides the decode lengths after the append;
    ``prefill`` = (prior, chunk) overrides the prefill chunk.  Decode
    sequence b stores its new token at position seq_lens_after[b] - 1; the
    prefill sequence stores its chunk at positions prior .. prior+chunk-1."""
    bs = w.block_size
    if seq_lens_after is None:
        seq_lens_after = context_lens(w) + 1
    seq_lens_after = torch.as_tensor(seq_lens_after, dtype=torch.int64)
    prior, chunk = prefill if prefill is not None else (w.prefill_prior, w.prefill_chunk)
    lengths = list(seq_lens_after.tolist())
    if chunk > 0:
        lengths.append(prior + chunk)
    nblk = [-(-n // bs) for n in lengths]
    used = sum(nblk)
    if w.pool_blocks:
        assert w.pool_blocks >= used
        num_blocks = w.pool_blocks
    else:
        num_blocks = used + int(math.ceil(used * w.spare_frac))
    g = torch.Generator().manual_seed(2000 + w.seed + seed_offset)
    perm = torch.randperm(num_blocks, generator=g)
    max_blocks = max(nblk) if nblk else 1
    # tail entries: valid ids of unrelated blocks (never to be read)
    table = torch.randint(0, num_blocks, (len(lengths), max_blocks), generator=g)
    off = 0
    for r, n in enumerate(nblk):
        table[r, :n] = perm[off:off + n]
        off += n
    table = table.to(torch.int32)
    slots = []
    for b, n in enumerate(seq_lens_after.tolist()):
        p = n - 1
        slots.append(int(table[b, p // bs]) * bs + p % bs)
    if chunk > 0:
        r = len(lengths) - 1
        for p in range(prior, prior + chunk):
            slots.append(int(table[r, p // bs]) * bs + p % bs)
    return Layout(
        seq_lens=seq_lens_after.to(torch.int32), block_table=table, num_blocks=num_blocks,
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        num_decode_tokens=len(seq_lens_after), prefill_row=(len(lengths) - 1) if chunk > 0 else -1,
        used_blocks=used)


def _randn(shape, dtype, device, gen):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


@dataclass
class LayerInputs:
    q_decode: torch.Tensor    # [B, Hq, D]
    q_prefill: torch.Tensor   # [C, Hq, D] (C may be 0)
    k_new: torch.Tensor       # [T, Hkv, D]
    v_new: torch.Tensor       # [T, Hkv, D]
    k_cache: torch.Tensor     # [NB, Hkv, bs, D] before the append
    v_cache: torch.Tensor


def draw_layer(w: Workload, lay: Layout, layer: int = 0, device="cpu", with_pool: bool = True,
               dtype=None) -> LayerInputs:
    """N(0,1) inputs of one layer, seeded by (workload seed, layer)."""
    dtype = dtype or w.dtype
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(10_000 * (w.seed + 1) + layer)
    hq, hkv, d, bs = w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    t = lay.slot_mapping.shape[0]
    b = lay.num_decode_tokens
    c = t - b
    q_dec = _randn((b, hq, d), dtype, dev, gen)
    q_pre = _randn((c, hq, d), dtype, dev, gen)
    k_new = _randn((t, hkv, d), dtype, dev, gen)
    v_new = _randn((t, hkv, d), dtype, dev, gen)
    if with_pool:
        kc = _randn((lay.num_blocks, hkv, bs, d), dtype, dev, gen)
        vc = _randn((lay.num_blocks, hkv, bs, d), dtype, dev, gen)
    else:
        kc = vc = None
    return LayerInputs(q_dec, q_pre, k_new, v_new, kc, vc)


def sample_pairs(n_rows: int, n_heads: int, count: int, seed: int, must=()) -> list:
    """Seeded sample of (row, head) pairs, always including ``must`` rows
    (each with a seeded head)."""
    g = torch.Generator().manual_seed(30_000 + seed)
    pairs = {(int(r), int(torch.randint(0, n_heads, (1,), generator=g))) for r in must
             if 0 <= r < n_rows}
    while len(pairs) < min(count, n_rows * n_heads):
        r = int(torch.randint(0, n_rows, (1,), generator=g))
        h = int(torch.randint(0, n_heads, (1,), generator=g))
        pairs.add((r, h))
    return sorted(pairs)


def fp8_scales(w: Workload, layer: int = 0) -> tuple:
    """Seeded per-KV-head float32 scales (k_scale, v_scale) for an fp8 cache:
    a head's N(0,1) entries beyond 4 to 6 standard deviations saturate."""
    g = torch.Generator().manual_seed(50_000 + 100 * w.seed + layer)
    k = (4.0 + 2.0 * torch.rand(w.num_kv_heads, generator=g)) / 448.0
    v = (4.0 + 2.0 * torch.rand(w.num_kv_heads, generator=g)) / 448.0
    return k.to(torch.float32), v.to(torch.float32)


def draw_fp8_pool(w: Workload, lay: Layout, scales: torch.Tensor, layer: int = 0, which: int = 0,
                  device="cpu") -> torch.Tensor:
    """uint8 E4M3 codes [NB, Hkv, bs, D] standing for a cache of N(0,1)
    entries stored at ``scales`` [Hkv] (codes drawn through torch's own
    float8_e4m3fn cast, clamped to the finite range)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(20_000 * (w.seed + 1) + 2 * layer + which)
    x = torch.randn((lay.num_blocks, w.num_kv_heads, w.block_size, w.head_dim), generator=gen,
                    device=dev, dtype=torch.float32)
    x = (x / scales.to(dev)[None, :, None, None]).clamp_(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


@dataclass
class LatentInputs:
    q: torch.Tensor        # [B, Hq, D] bf16 (the decode queries)
    c_new: torch.Tensor    # [B, r] bf16 (each sequence's new token's latent)
    pool: torch.Tensor     # [NB, bs, r] bf16 latent pool before the append
    w_k: torch.Tensor      # [Hq, D, r] bf16 key up-projections
    w_v: torch.Tensor      # [Hq, D, r] bf16 value up-projections


def draw_latent(w: Workload, lay: Layout, rank: int = 128, layer: int = 0,
                device="cpu") -> LatentInputs:
    """Seeded inputs of the latent (MLA-style) cache for the decode batch of
    ``lay``: N(0,1) queries and latents, and up-projections with N(0, 1/r)
    entries, so reconstructed keys and values have unit variance."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(30_000 * (w.seed + 1) + layer)
    b = lay.num_decode_tokens
    q = _randn((b, w.num_q_heads, w.head_dim), torch.bfloat16, dev, gen)
    c_new = _randn((b, rank), torch.bfloat16, dev, gen)
    pool = _randn((lay.num_blocks, w.block_size, rank), torch.bfloat16, dev, gen)
    s = 1.0 / math.sqrt(rank)
    w_k = (torch.randn((w.num_q_heads, w.head_dim, rank), generator=gen, device=dev) * s).to(torch.bfloat16)
    w_v = (torch.randn((w.num_q_heads, w.head_dim, rank), generator=gen, device=dev) * s).to(torch.bfloat16)
    return LatentInputs(q, c_new, pool, w_k, w_v)
