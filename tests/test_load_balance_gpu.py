"""Load balance of the tensor-core forward (advanced load balancing for skew:
longest-first claiming).

The forward.rs page walks its WorkSplit list with a thread pool; here the
units (kv head, block) are claimed by persistent CTAs from a counter that
walks a list with the heavy units (a thirty-second of a CTA's mean share of edges
or more) first, by descending size class, and the light rest in index
order.  On a skewed selection
(Zipf block popularity: a few units with hundreds of edges, many with a few)
the test reads back each CTA's claimed rows and busy cycles
(sa_debug_cta_stats) with the longest-first list and with plain index order,
and checks that the longest-first schedule is balanced and that the results
are bit-identical (a unit's partials do not depend on which CTA runs it).
"""
import numpy as np
import pytest
import torch

import _gpu
import block_sparse_paged_csr_gb300 as sa
import inputs

pytestmark = pytest.mark.gpu


def _forward_with_stats(w, t, index, n_ctas, lpt):
    keep = index.c.workspace_bytes
    if not lpt:
        index.c.workspace_bytes = 256        # room for the counter only: index order
    stats = torch.zeros(3 * n_ctas, dtype=torch.int64, device="cuda")
    sa.sa_debug_cta_stats(stats)
    try:
        o, m, l = sa.sa_forward(t["q"], t["k"], t["v"], index, t["bt"], t["cu"], t["used"], w.hq,
                                w.hkv, w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                                w.causal)
        torch.cuda.synchronize()
    finally:
        sa.sa_debug_cta_stats(None)
        index.c.workspace_bytes = keep
    assert sa.sa_get_status(index) == 0
    s = stats.view(n_ctas, 3).cpu().numpy()
    return (o, m, l), s


def test_longest_first_claiming_balances_the_skewed_forward():
    w = inputs.skewed(0, batch=4)
    assert _gpu.auto_uses_tensor_cores(w)
    t = _gpu.device_workload(w, fill_on_device=True)
    index = sa.sa_build_index(t["selected"], w.cu_seqlens_q, t["cu"], t["used"], w.max_pages,
                              w.block_size, w.page_size)
    n_ctas = torch.cuda.get_device_properties(0).multi_processor_count
    results = {}
    for lpt in (True, False):
        _forward_with_stats(w, t, index, n_ctas, lpt)              # warm-up
        parts, s = _forward_with_stats(w, t, index, n_ctas, lpt)
        rows, units, cycles = s[:, 0], s[:, 1], s[:, 2]
        busy = cycles > 0
        assert busy.sum() == min(n_ctas, int(units.sum()))
        assert int(units.sum()) == int(index.totals[2])             # every unit once
        assert int(rows.sum()) == int(index.totals[0]) * w.qhead    # every row once
        results[lpt] = (parts, rows[busy].max() / rows[busy].mean(),
                        cycles[busy].max() / cycles[busy].mean())
    (p1, r1, c1), (p0, r0, c0) = results[True], results[False]
    for a, b in zip(p1, p0):
        n = int(index.totals[0]) * w.qhead
        assert torch.equal(a[:n], b[:n]), "partials depend on the claim order"
    _gpu.REPORT.append(("balance skewed(batch 4): longest-first", "rows,cyc", float(r1),
                        float(c1)))
    _gpu.REPORT.append(("balance skewed(batch 4): index order", "rows,cyc", float(r0),
                        float(c0)))
    assert c1 <= 1.05, f"busy-cycle max/mean {c1:.3f} with the longest-first list"
    assert c1 <= c0 + 0.01
