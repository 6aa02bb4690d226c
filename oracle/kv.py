"""CPU oracle of the KV-cache commit after verification (test infrastructure
only).

Source: the "Speculative Decoding and EAGLE-3" lesson, section "KV cache
rollback": the verify pass extends the verifier's KV cache by the window's
entries; after a rejection at position j the entries past the correction are
wrong, and there are two common implementations -- write the window to a
scratch buffer and commit the accepted entries on acceptance (vLLM,
TensorRT-LLM), or keep the physical cache and a separate logical length that
is cut back on rejection; exercise 4 (two sequences, one accepting every
draft and one rejecting at position 2, each with its own correct
kv_length).  The committed count is the verify step's out_kv_len
(= accepted + 1: the verified input token's entry plus the accepted drafts).

Readings of points the pages leave open:

* Layout: the cache is [L, B, S, E] (L layers, B sequences, S positions, E
  bytes per position and layer: all heads' keys and values); the scratch
  window is [L, B, W, E].  seq_len[b] is the logical length before the
  commit.
* Kept window positions: 0 (the verified input token), then for a chain
  1, 2, ..., and for a tree the accepted node ids out_path[b, :], in that
  order; kv_len[b] of them in all (kv_len <= 0: a failed request, nothing
  kept, the length unchanged).
* SCRATCH mode copies kept position i of the window to cache position
  seq_len + i.  IN-PLACE mode assumes the verify pass wrote window position
  w at cache position seq_len + w and moves kept position i from
  seq_len + pos_i to seq_len + i (nothing moves for a chain).  Either way
  seq_len becomes seq_len + kv_len; entries past the new length are left as
  they are (the logical length is what hides them).
* A commit that would pass S, read a window position outside the window,
  or keep positions that do not rise (a walk's path always rises: a child's
  id exceeds its parent's) is refused for that sequence: cache and length
  unchanged, error bit ERR_KV.
"""

import numpy as np

SCRATCH = 0
INPLACE = 1
ERR_KV = 16


def kept_positions(kv_len, path=None):
    """Window positions whose entries are kept, in cache order."""
    if kv_len <= 0:
        return []
    if path is None:
        return list(range(kv_len))
    return [0] + [int(x) for x in path[:kv_len - 1]]


def commit(mode, cache, seq_len, kv_len, scratch=None, path=None):
    """Commit every sequence's kept entries.  cache [L, B, S, E] (uint8) is
    updated in place and returned with the new lengths and the OR of error
    bits."""
    L, B, S, E = cache.shape
    seq_len = np.asarray(seq_len, dtype=np.int64).copy()
    errors = 0
    for b in range(B):
        n = int(kv_len[b])
        if n <= 0:
            continue
        pos = kept_positions(n, None if path is None else path[b])
        start = int(seq_len[b])
        width = scratch.shape[2] if mode == SCRATCH else S - start
        rising = all(pos[i] > pos[i - 1] for i in range(1, len(pos)))
        if start < 0 or start + n > S or len(pos) != n or min(pos) < 0 or max(pos) >= width \
                or not rising:
            errors |= ERR_KV
            continue
        src = scratch[:, b] if mode == SCRATCH else cache[:, b, start:].copy()
        for i, w in enumerate(pos):
            cache[:, b, start + i, :] = src[:, w, :]
        seq_len[b] = start + n
    return cache, seq_len, errors


def bytes_moved(mode, kv_len, entry_bytes, layers, path=None):
    """Bytes read plus written by a commit (in-place entries that stay where
    they are cost nothing)."""
    total = 0
    for b, n in enumerate(np.asarray(kv_len).reshape(-1)):
        pos = kept_positions(int(n), None if path is None else path[b])
        moved = len(pos) if mode == SCRATCH else sum(1 for i, w in enumerate(pos) if w != i)
        total += 2 * moved * entry_bytes * layers
    return total
