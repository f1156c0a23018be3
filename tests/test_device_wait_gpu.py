"""Bounded device waits run out cleanly (the pages' GpuRuntimeError, types.rs
error enum, stands for any device failure; here it is SA_ERR_DEVICE_TIMEOUT).

Each test makes one wait that nothing will ever satisfy (sa_debug_stall, a
test hook of the library) with a short spin limit, checks that the kernel
gives up, reports SA_ERR_DEVICE_TIMEOUT through sa_get_status and returns
(no hang, no fault), and then that the next clean call on the same context
reports OK and matches the oracle.  No wait is removed and no copy is left
in flight: the index kernel's grid barrier is simply never released, or the
fused decode kernel's load warps issue no copy.
"""
import numpy as np
import pytest

import _gpu
import block_sparse_paged_csr_gb300 as sa
import inputs
import oracle

pytestmark = pytest.mark.gpu

SPIN = 2000


def _check_clean_call(w, t):
    out, lse, idx, _ = _gpu.run_attention(w, t)      # asserts status OK
    ref, ref_lse, ref_idx, _ = oracle.attention(w.q_host(), w.k_host(), w.v_host(), w.selected,
                                                w.block_tables, w.cu_seqlens_q, w.used, w.hq,
                                                w.head_dim, w.block_size, w.page_size,
                                                w.softmax_scale, w.causal)
    _gpu.compare_index(idx.to_host(), ref_idx)
    assert _gpu.row_error(out.cpu().numpy(), ref) <= _gpu.auto_tol(w)


@pytest.mark.parametrize("site,name", [(sa.STALL_INDEX_BARRIER, "gqa_decode"),
                                       (sa.STALL_FUSED_COPIES, "gqa_decode"),
                                       (sa.STALL_FUSED_COPIES, "long_decode")])
def test_bounded_wait_runs_out_and_the_next_call_is_clean(site, name):
    w = inputs.small(name, seed=4)
    t = _gpu.device_workload(w)
    # both stall sites sit on the fused decode path (which reads no output of
    # the index kernel, so an unfinished index is never dereferenced)
    assert _gpu.uses_fused(w)
    sa.sa_debug_stall(site, SPIN)
    try:
        _, _, idx, _ = sa.sa_attention(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q,
                                       t["cu"], t["used"], t["bt"], w.hq, w.hkv, w.head_dim,
                                       w.block_size, w.page_size, w.softmax_scale, w.causal)
        status = sa.sa_get_status(idx)
    finally:
        sa.sa_debug_stall(sa.STALL_NONE, 0)
    assert sa.sa_status_string(status) == sa.sa_status_string(9)
    assert status == 9, f"expected DEVICE_TIMEOUT, got {status}"
    _check_clean_call(w, t)


def test_debug_stall_rejects_unknown_sites():
    with pytest.raises(sa.SAError, match="INVALID_ARGUMENT"):
        sa.sa_debug_stall(7, 0)
