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
