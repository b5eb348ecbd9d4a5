"""Planner oracle: common-prefix length and the pages' use-cascade thresholds.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  Pure-Python loops over the block table,
written for reading, not for speed.

Sources
-------
* "vLLM Cascade Attention：用法、场景与原理解析" (beaiera.top)
  - §八 Step 1: scan the block tables of all running requests and count the
    physical blocks they share, matching consecutively from block 0.
  - §八 Step 2: common_prefix_len = blocks * block_size, capped to the minimum
    num_computed_tokens, then floored to a multiple of block_size.
  - §四: the cap keeps the prefix inside every request's already-computed KV,
    so the non-causal prefix phase cannot leak later tokens (the R1/R2 example).
  - §三: the use-cascade thresholds, prefix >= 256 tokens and batch >= 8 requests.
* "fix(v1/kv_cache): resolve async KV transfer bug in cascade attention #23485":
  only requests that are actually running take part; the planner is handed
  exactly those rows and nothing else.

Reading where the pages are silent: entries of a row past cdiv(seq_len, block_size)
are padding and never take part in the match (a row can only share blocks it uses).
"""

from __future__ import annotations


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def num_common_prefix_blocks(block_table, seq_lens, block_size: int) -> int:
    """Longest run, from block 0, of identical physical block ids in every row.

    block_table: sequence of rows (any indexable of ints); seq_lens: KV length per
    request.  Rows take part only up to their own cdiv(seq_len, block_size) blocks.
    Zero requests share nothing.
    """
    n = len(seq_lens)
    if n == 0:
        return 0
    used = [_cdiv(int(seq_lens[r]), block_size) for r in range(n)]
    k = 0
    while True:
        if any(k >= used[r] for r in range(n)):
            return k
        first = int(block_table[0][k])
        if any(int(block_table[r][k]) != first for r in range(n)):
            return k
        k += 1


def common_prefix_len(num_blocks_shared: int, block_size: int, num_computed_tokens) -> int:
    """§八 Step 2: blocks to tokens, cap to min(num_computed_tokens), floor to block_size."""
    if len(num_computed_tokens) == 0:
        return 0
    cpl = num_blocks_shared * block_size
    cpl = min(cpl, min(int(x) for x in num_computed_tokens))
    cpl = (cpl // block_size) * block_size
    return cpl


def use_cascade_thresholds(cpl: int, num_reqs: int) -> bool:
    """§三 thresholds only: prefix of at least 256 tokens and at least 8 requests."""
    return cpl >= 256 and num_reqs >= 8


def plan(block_table, seq_lens, num_computed_tokens, block_size: int):
    """(common_prefix_len, use_cascade by the pages' thresholds) for one batch."""
    ncpb = num_common_prefix_blocks(block_table, seq_lens, block_size)
    cpl = common_prefix_len(ncpb, block_size, num_computed_tokens)
    return cpl, use_cascade_thresholds(cpl, len(seq_lens))


# -- multi-level cascade ---------------------------------------------------------------
# "vLLM Cascade Attention：用法、场景与原理解析" §七: FlashInfer's cascade runs any
# number of levels (num_levels), where vLLM's runs two (prefix + suffix).  Reading: the
# levels form a prefix tree over consecutive requests; a level-d segment is a run of at
# least two consecutive requests that share the blocks of keys [k_lo, k_hi) beyond the
# segment of level d - 1 that holds them (level 0: the whole batch, from key 0).  Within
# each segment the plan is §八 Step 1-2's again: the longest run of shared block ids from
# k_lo (each row only within its used entries), capped to the segment's minimum
# num_computed_tokens and floored to block_size; a request's suffix starts at the end of
# the deepest segment that holds it.  Below a segment, the requests split into maximal
# runs that share the next block; a run of one request has no further level.


def plan_levels(block_table, seq_lens, num_computed_tokens, block_size: int,
                max_levels: int):
    """(segments, suffix_start): segments as (level, r_lo, r_hi, k_lo, k_hi) in the order
    a depth-first walk emits them, and each request's suffix start (token)."""
    n = len(seq_lens)
    used = [_cdiv(int(seq_lens[r]), block_size) for r in range(n)]
    start = [0] * n
    segments = []

    def shared_run(r_lo, r_hi, col):
        """Columns from `col` on that every row of [r_lo, r_hi) uses and shares."""
        k = col
        while True:
            if any(k >= used[r] for r in range(r_lo, r_hi)):
                return k - col
            first = int(block_table[r_lo][k])
            if any(int(block_table[r][k]) != first for r in range(r_lo, r_hi)):
                return k - col
            k += 1

    def walk(r_lo, r_hi, k_lo, level):
        if level >= max_levels:
            return
        k_next = k_lo
        if r_hi - r_lo >= 2:
            nb = shared_run(r_lo, r_hi, k_lo // block_size)
            k_hi = (k_lo // block_size + nb) * block_size
            k_hi = min(k_hi, min(int(num_computed_tokens[r]) for r in range(r_lo, r_hi)))
            k_hi = (k_hi // block_size) * block_size
            if k_hi > k_lo:
                segments.append((level, r_lo, r_hi, k_lo, k_hi))
                for r in range(r_lo, r_hi):
                    start[r] = k_hi
                k_next = k_hi
        # the runs of consecutive requests that share the block at k_next
        col = k_next // block_size
        r = r_lo
        while r < r_hi:
            e = r + 1
            if col < used[r]:
                while e < r_hi and col < used[e] and \
                        int(block_table[e][col]) == int(block_table[r][col]):
                    e += 1
            if e - r >= 2 and not (r == r_lo and e == r_hi and k_next == k_lo):
                walk(r, e, k_next, level + 1)
            r = e

    if n > 0:
        walk(0, n, 0, 0)
    return segments, start
