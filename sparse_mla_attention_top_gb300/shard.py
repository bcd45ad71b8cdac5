"""Token-sharded prefill across ranks (the pages' ShardQ layout), as host-side partitions.

vLLM PR #63104, Overview: under tensor parallelism each rank takes a slice of the prefill
tokens with every head, token-major, so 128 / H consecutive tokens of the slice fill one
packed row; the slices are "zigzag" chunks (the rank's bench script): the tokens are cut
into 2 * world near-equal chunks and rank r takes chunk r and chunk 2 * world - 1 - r, one
early and one late, which evens out the causal work (late tokens see longer prefixes).

Each rank then runs the ordinary grouped prefill on its own rows: its q and top-k rows are
the selected tokens' rows, and a group may straddle the two chunks, since every query keeps
to its own entries through its membership bit. No data moves between ranks; the outputs of
all ranks together are the whole step's outputs, row for row.
"""

from __future__ import annotations

import numpy as np


def zigzag_split(n_tokens: int, world: int) -> list:
    """Token ids (ascending int64 arrays) of each rank; together they cover 0..n-1 once."""
    if world < 1 or n_tokens < 0:
        raise ValueError("world must be >= 1 and n_tokens >= 0")
    bounds = np.linspace(0, n_tokens, 2 * world + 1).round().astype(np.int64)
    chunks = [np.arange(bounds[i], bounds[i + 1], dtype=np.int64) for i in range(2 * world)]
    return [np.concatenate([chunks[r], chunks[2 * world - 1 - r]]) for r in range(world)]
