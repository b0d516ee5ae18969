"""Seeded packed-row layouts for the packed-row tests: rows of consecutive
documents drawn from random lengths, as an indexed packing mask and as the
two row-local arrays of flatten_packed_sequence_metadata. Holds no
conversion arithmetic: the flat outputs come from the oracle."""

import numpy as np


def packed_rows(seed, b=6, s=40, max_docs=5, max_doc_len=12, sparse=False):
    """Returns (ids [b, s] int32, token_indices [b, s] int64, row_cu [b, max_docs+1] int32)."""
    rng = np.random.default_rng(seed)
    ids = np.zeros((b, s), np.int32)
    tok = np.full((b, s), -1, np.int64)
    rcu = np.full((b, max_docs + 1), -1, np.int32)
    for i in range(b):
        docs, room = [], s
        for _ in range(int(rng.integers(0, max_docs + 1))):
            if room == 0:
                break
            docs.append(int(rng.integers(1, min(room, max_doc_len) + 1)))
            room -= docs[-1]
        n = sum(docs)
        ids[i, :n] = np.repeat(np.arange(1, len(docs) + 1), docs)
        tok[i, :n] = np.sort(rng.choice(s, n, replace=False)) if sparse else np.arange(n)
        rcu[i, :len(docs) + 1] = np.concatenate([[0], np.cumsum(docs)])
    return ids, tok, rcu
