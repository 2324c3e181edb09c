"""Synthetic prompts.

``uniform_prompt``: i.i.d. uniform token ids (the tiny, 0.5B and 7B workloads).

``ngram_prompt``: the prompt-lookup workload. A seeded base sequence of
uniform tokens is drawn; the prompt is then built left to right out of
segments of length U{16..64}. With probability ``r`` a segment copies a
random span of that length out of the base sequence, otherwise it is fresh
uniform tokens. ``repeated_fraction`` reports the share of prompt tokens that
came from copied spans.
"""

import torch


def uniform_prompt(n: int, high: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, high, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def ngram_prompt(total: int, r: float, vocab: int, seed: int, base_len: int = 512,
                 seg_lo: int = 16, seg_hi: int = 64):
    """Returns (prompt int32 [total], copied mask bool [total])."""
    g = torch.Generator().manual_seed(seed)
    base = torch.randint(0, vocab, (base_len,), generator=g, dtype=torch.int64)
    toks, mask = [], []
    n = 0
    while n < total:
        seg = int(torch.randint(seg_lo, seg_hi + 1, (1,), generator=g))
        seg = min(seg, total - n)
        if float(torch.rand((1,), generator=g)) < r:
            start = int(torch.randint(0, base_len - seg + 1, (1,), generator=g))
            toks.append(base[start:start + seg])
            mask.append(torch.ones(seg, dtype=torch.bool))
        else:
            toks.append(torch.randint(0, vocab, (seg,), generator=g, dtype=torch.int64))
            mask.append(torch.zeros(seg, dtype=torch.bool))
        n += seg
    return torch.cat(toks).to(torch.int32), torch.cat(mask)


def repeated_fraction(mask: torch.Tensor) -> float:
    return float(mask.float().mean())
