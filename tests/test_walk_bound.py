"""The partial-slot bound behind the decode workspace, on a model of the
balanced walk's share arithmetic (no GPU).

The decode kernels flatten every stream's stages into one list of S stages
and give CTA c the stages [c*S/C, (c+1)*S/C) of it (integer division), but
only when S >= (512 / stage_tokens) * C, so every share holds at least 512
tokens of stages.  A stream is (sequence, KV head) with 64-token stages, or
(sequence, group of four KV heads) with 16-token stages.  The workspace has
ceil(max_len / 512) + 1 partial slots per row, so a stream of n tokens must
fall to at most ceil(n / 512) + 1 CTAs for every partial index to stay in
bounds.  This checks that bound on random batches and grids, for both stage
sizes, and that the shares tile the list exactly."""
import random

import pytest

SPLIT = 512


def shares(total, ctas):
    return [(c * total // ctas, (c + 1) * total // ctas) for c in range(ctas)]


@pytest.mark.parametrize("stage_tokens,streams_per_seq", [(64, 8), (64, 2), (16, 2), (16, 1)])
def test_pieces_per_stream_fit_the_partial_slots(stage_tokens, streams_per_seq):
    rng = random.Random(1234 + stage_tokens + streams_per_seq)
    checked = 0
    for _ in range(300):
        nseq = rng.randint(1, 160)
        lens = [max(1, int(rng.choice([rng.uniform(1, 600), rng.expovariate(1 / 6000)])))
                for _ in range(nseq)]
        ctas = rng.choice([152, 304, 327, 330, 456, rng.randint(1, 600)])
        streams = []                     # (first stage, stages, tokens)
        pos = 0
        for n in lens:
            st = -(-n // stage_tokens)
            for _ in range(streams_per_seq):
                streams.append((pos, st, n))
                pos += st
        total = pos
        if total < (SPLIT // stage_tokens) * ctas:
            continue                     # the kernels take 512-token splits here
        sh = shares(total, ctas)
        assert sh[0][0] == 0 and sh[-1][1] == total
        assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
        assert min(e - b for b, e in sh) * stage_tokens >= SPLIT
        for first, st, n in streams:
            pieces = sum(1 for b, e in sh if b < first + st and e > first)
            assert pieces <= -(-n // SPLIT) + 1, (n, pieces)
        checked += 1
    assert checked > 50


def test_split_walk_units_fit_the_partial_slots():
    """512-token splits: a stream of n tokens has exactly ceil(n / 512) units."""
    for n in (1, 511, 512, 513, 1024, 32769):
        units = [(s, min(n, s + SPLIT)) for s in range(0, n, SPLIT)]
        assert len(units) == -(-n // SPLIT)
        assert units[-1][1] == n and all(e - b <= SPLIT for b, e in units)


def test_latent_walk_with_padding_fits_the_partial_slots():
    """The latent decode's walk: 128-token stages, four empty stages counted
    after each sequence's real ones, shares of at least four stages.  The
    padding follows the real stages, so the real ones still fall to at most
    ceil(n / 512) + 1 CTAs."""
    rng = random.Random(77)
    stage, pad, min_stages = 128, 4, SPLIT // 128
    checked = 0
    for _ in range(300):
        lens = [max(1, int(rng.expovariate(1 / rng.choice([300, 3000, 12000]))))
                for _ in range(rng.randint(1, 160))]
        ctas = rng.choice([148, 152, rng.randint(1, 400)])
        streams, pos = [], 0
        for n in lens:
            real = -(-n // stage)
            streams.append((pos, real, n))
            pos += real + pad
        if pos < min_stages * ctas:
            continue
        sh = shares(pos, ctas)
        for first, real, n in streams:
            pieces = sum(1 for b, e in sh if b < first + real and e > first)
            assert pieces <= -(-n // SPLIT) + 1, (n, pieces)
        checked += 1
    assert checked > 50
