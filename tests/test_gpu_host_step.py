"""GPU parity of cascade_step_host: a whole step from (pinned) host buffers — copies in,
host planner, attention call, copies out — against the oracle."""

import numpy as np
import pytest
import torch

from shared_prefix_paged_gb300 import csp, workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _host_step(b, mode, scratch=None):
    pin = lambda t: t.contiguous().pin_memory()
    q = pin(b.q)
    bt = pin(torch.from_numpy(np.ascontiguousarray(b.block_table)))
    cu = pin(torch.from_numpy(b.cu_seqlens_q))
    sl = pin(torch.from_numpy(b.seq_lens))
    nc = pin(torch.from_numpy(b.num_computed_tokens))
    out = torch.full(b.q.shape, 7.0, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((b.total_q, b.num_q_heads), dtype=torch.float32).pin_memory()
    k, v = b.k_cache.cuda(), b.v_cache.cuda()
    cpl, _ = csp.cascade_plan(b.block_table, b.seq_lens, b.num_computed_tokens,
                              block_size=b.block_size)
    if scratch is None:
        need = max(csp.step_scratch_size(b.cu_seqlens_q, b.seq_lens, b.block_table.shape[1], c,
                                         b.num_q_heads, b.num_kv_heads, b.head_dim)
                   for c in (0, cpl))
        scratch = csp.alloc_workspace(need, "cuda")
    step = csp.HostStep(q, bt, cu, sl, nc, k, v, softmax_scale=b.scale, out=out, lse=lse,
                        scratch=scratch, mode=mode)
    used = step()
    return out, lse, used, cpl


@pytest.mark.parametrize("mode", [csp.MODE_FORCE_CASCADE, csp.MODE_FORCE_FLAT])
@pytest.mark.parametrize("name", ["tiny", "chunked"])
def test_host_step_all_rows(name, mode):
    b = workloads.by_name(name)
    ref_o, ref_l = H.oracle_ref(b)
    out, lse, used, cpl = _host_step(b, mode)
    assert used == (cpl if mode == csp.MODE_FORCE_CASCADE else 0)
    H.compare(out, lse, ref_o, ref_l, what=f"host step {name} mode {mode}")


def test_host_step_decode_sampled_and_repeated():
    b = workloads.decode_batch()
    rows = H.sample_rows(b, 200, seed=77)
    ref_o, ref_l = H.oracle_ref(b, rows)
    for _ in range(3):   # the same scratch, the same host buffers, call after call
        out, lse, used, cpl = _host_step(b, csp.MODE_AUTO)
        assert used == cpl == 4096
        H.compare(out, lse, ref_o, ref_l, rows=rows, what="host step decode")


def test_host_step_scratch_too_small():
    b = workloads.tiny_decode()
    small = csp.alloc_workspace(1024, "cuda")
    with pytest.raises(csp.CspError) as e:
        _host_step(b, csp.MODE_FORCE_CASCADE, scratch=small)
    assert e.value.status == csp.CSP_ERR_WORKSPACE
