"""GPU parity of the single-kernel cascade schedule.

cascade_attn runs batches whose requests have at most 16 packed rows (query, head in
group) per KV head as one cooperative kernel: some CTAs run ranges of the prefix phase
on tcgen05 while the others stream suffix units (request, KV head) through a
producer warp's TMA ring, then every CTA merges a share of the rows after a grid-wide
barrier.  These cases
exercise that kernel's own logic against the oracle: causal suffix rows of several
queries, group sizes at the 16-row limit, D 64, suffixes of many tiles, a request
without queries, the fallback to two kernels, and one workspace reused across calls
of different shapes (its barrier count grows by the grid on every single-kernel call).
"""

import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def small(seed, seq, ql, shared, hq, hkv, d):
    g = torch.Generator().manual_seed(seed)
    return workloads.build_batch(f"single{seed}", seq, ql, shared, num_q_heads=hq,
                                 num_kv_heads=hkv, head_dim=d, gen=g)


def schedule(b, cpl):
    return csp.cascade_schedule(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, cpl,
                                b.num_q_heads, b.num_kv_heads, b.head_dim)


# (seed, seq_lens, q_lens, shared tokens, Hq, Hkv, D)
CASES = [
    (31, [300, 320, 350, 310], [4, 3, 1, 2], 288, 32, 8, 128),        # causal rows, group 4
    (32, [400, 420, 401], [1, 1, 1], 384, 32, 2, 128),                # group 16: 16 rows
    (33, [200, 230, 260, 290], [16, 7, 1, 12], 160, 4, 4, 64),        # group 1, 16 rows, D 64
    (34, [700] * 9, [1] * 9, 640, 16, 2, 64),                         # D 64, group 8
    (35, [2000, 2100, 1900], [1, 2, 1], 1024, 8, 2, 128),             # suffix ~1000 keys
    (36, [272, 600, 301, 288, 1000], [1, 1, 2, 1, 1], 272, 16, 4, 128),  # ragged suffixes
]


SINGLE = dict(schedule=csp.SCHEDULE_SINGLE)


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_single_kernel_all_rows(case):
    # the schedule is forced: with few long suffixes the cost model would rather take
    # the two-kernel schedule, but these shapes exercise the single kernel's own paths
    seed, seq, ql, shared, hq, hkv, d = case
    b = small(seed, seq, ql, shared, hq, hkv, d)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    assert cpl > 0
    out, lse = H.run_cascade(b, dev, cpl, **SINGLE)
    H.compare(out, lse, ref_o, ref_l, what="single kernel")
    # a shorter prefix is as valid: more of each request's keys go to the suffix phase
    out, lse = H.run_cascade(b, dev, 16, **SINGLE)
    H.compare(out, lse, ref_o, ref_l, what="single kernel cpl=16")
    # other numbers of prefix ranges (one range; several, with prefix CTAs taking units)
    for r in (1, 3):
        out, lse = H.run_cascade(b, dev, cpl, prefix_ranges=r, **SINGLE)
        H.compare(out, lse, ref_o, ref_l, what=f"single kernel, {r} prefix ranges")


def test_forced_schedules_and_errors():
    b = small(38, [300, 320, 350, 310], [4, 3, 1, 2], 288, 32, 8, 128)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    out, lse = H.run_cascade(b, dev, cpl, schedule=csp.SCHEDULE_TWO_KERNELS)
    H.compare(out, lse, ref_o, ref_l, what="forced two kernels")
    with pytest.raises(csp.CspError) as e:
        H.run_cascade(b, dev, cpl, schedule=7)
    assert e.value.status == csp.CSP_ERR_INVALID_ARG
    # 16 query tokens x group 4: 64 rows per request and KV head, past the 16-row tile
    wide = small(39, [300, 310], [16, 16], 288, 32, 8, 128)
    wdev = H.to_device(wide)
    wcpl, _ = H.plan(wide, mode=csp.MODE_FORCE_CASCADE)
    with pytest.raises(csp.CspError) as e:
        H.run_cascade(wide, wdev, wcpl, **SINGLE)
    assert e.value.status == csp.CSP_ERR_UNSUPPORTED


def test_cost_model_picks_single_kernel_for_decode():
    b = workloads.decode_batch()
    assert schedule(b, 4096)[0] == csp.SCHEDULE_SINGLE


def test_request_without_queries():
    b = small(37, [300, 310, 305, 330], [1, 0, 2, 1], 288, 8, 2, 128)
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
    out, lse = H.run_cascade(b, dev, cpl, **SINGLE)
    H.compare(out, lse, ref_o, ref_l, what="empty request")


def test_last_block_with_one_m_tile():
    # 80 requests x group 4 = 320 packed rows per KV head: blocks of 256 + 64 rows
    b = workloads.decode_batch(seed=3101, n=80, p=512, s=40)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 800, seed=1)
    ref_o, ref_l = H.oracle_ref(b, rows)
    cpl, _ = H.plan(b)
    out, lse = H.run_cascade(b, dev, cpl, **SINGLE)
    H.compare(out, lse, ref_o, ref_l, rows, what="N=80")


def test_too_many_prefix_blocks_falls_back():
    # 1024 requests x group 16 = 64 blocks of 256 rows per KV head, 4 KV heads: more
    # prefix blocks than SMs, so the two-kernel schedule runs
    b = workloads.decode_batch(seed=3102, n=1024, p=256, s=24, num_q_heads=64,
                               num_kv_heads=4, head_dim=64)
    dev = H.to_device(b)
    rows = H.sample_rows(b, 1000, seed=2)
    ref_o, ref_l = H.oracle_ref(b, rows)
    cpl, _ = H.plan(b)
    assert cpl == 256
    assert schedule(b, cpl)[0] == csp.SCHEDULE_TWO_KERNELS
    out, lse = H.run_cascade(b, dev, cpl)
    H.compare(out, lse, ref_o, ref_l, rows, what="N=1024 group 16")


def test_one_workspace_across_shapes():
    batches = [workloads.tiny_decode(), small(38, [300, 320, 350, 310], [4, 3, 1, 2], 288,
                                              32, 8, 128), workloads.tiny_decode(seed=1005)]
    prepared = []
    need = 0
    for b in batches:
        cpl, _ = H.plan(b, mode=csp.MODE_FORCE_CASCADE)
        need = max(need, csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q,
                                            b.max_seqlen_k, cpl, b.num_q_heads,
                                            b.num_kv_heads, b.head_dim))
        prepared.append((b, H.to_device(b), cpl, H.oracle_ref(b)))
    ws = csp.alloc_workspace(need, torch.device("cuda"))
    for _ in range(3):
        for b, dev, cpl, (ref_o, ref_l) in prepared:
            out, lse = H.run_cascade(b, dev, cpl, workspace=ws)
            H.compare(out, lse, ref_o, ref_l, what=b.name)
    assert csp.workspace_status(ws) == csp.CSP_OK
    # the single-kernel schedule's barrier count (header bytes [64, 72), 64-bit) grew by
    # the grid, one CTA per SM, on each of its calls and on nothing else
    singles = sum(3 for b, _, cpl, _ in prepared if schedule(b, cpl)[0] == csp.SCHEDULE_SINGLE)
    assert singles > 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    count = int(ws[64:72].cpu().view(torch.int64).item())
    assert count == singles * sms


def test_timed_variant_runs_the_same_kernel():
    b = workloads.tiny_decode()
    dev = H.to_device(b)
    ref_o, ref_l = H.oracle_ref(b)
    cpl, _ = H.plan(b)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in events:
        e.record()
    out, lse = H.run_cascade(b, dev, cpl, phase_events=events)
    H.compare(out, lse, ref_o, ref_l, what="timed")
    torch.cuda.synchronize()
    assert events[0].elapsed_time(events[1]) > 0
