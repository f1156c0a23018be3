"""sa_attention's fused decode path runs the index build on a side stream
beside the fused kernel and joins it back before it returns.  Checked here:
calls on a caller-created stream, back-to-back calls whose inputs change in
between, and two host threads with their own streams, each against the
oracle (output and the index, bit for bit)."""
import threading

import numpy as np
import pytest
import torch

import _gpu
import block_sparse_paged_csr_gb300 as sa
import inputs
import oracle

pytestmark = pytest.mark.gpu


def _attention(w, t, **kw):
    return sa.sa_attention(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q, t["cu"],
                           t["used"], t["bt"], w.hq, w.hkv, w.head_dim, w.block_size, w.page_size,
                           w.softmax_scale, w.causal, **kw)


def _reference(w, q_host, selected):
    return oracle.attention(q_host, w.k_host(), w.v_host(), selected, w.block_tables,
                            w.cu_seqlens_q, w.used, w.hq, w.head_dim, w.block_size, w.page_size,
                            w.softmax_scale, w.causal)


def _check(w, out, idx, q_host, selected):
    ref, _, ref_idx, _ = _reference(w, q_host, selected)
    _gpu.compare_index(idx.to_host(), ref_idx)
    assert _gpu.row_error(out.cpu().numpy(), ref) <= _gpu.auto_tol(w)


@pytest.mark.parametrize("name", ["gqa_decode", "long_decode"])
def test_calls_on_a_caller_stream_with_changing_inputs(name):
    w = inputs.small(name, seed=11)
    assert _gpu.uses_fused(w)
    t = _gpu.device_workload(w)
    stream = torch.cuda.Stream()
    rng = np.random.default_rng(5)
    with torch.cuda.stream(stream):
        out, lse, idx, parts = _attention(w, t)
        # a second call on the same buffers right behind the first, with new
        # queries and the ranks of every selection rotated (same blocks)
        q2 = rng.standard_normal(w.q_host().shape).astype(np.float32)
        sel2 = np.roll(w.selected, 1, axis=2)
        t["q"].copy_(torch.from_numpy(q2), non_blocking=False)
        t["selected"].copy_(torch.from_numpy(sel2))
        out, lse, idx, parts = _attention(w, t, index=idx, partials=parts, out=out, lse=lse)
    stream.synchronize()
    assert sa.sa_get_status(idx, stream=stream) == 0
    _check(w, out, idx, q2, sel2)


def test_two_threads_with_their_own_streams():
    cases = [inputs.small("gqa_decode", seed=21), inputs.small("long_decode", seed=22)]
    results = [None, None]
    errors = []

    def work(k):
        try:
            w = cases[k]
            t = _gpu.device_workload(w)
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for _ in range(5):
                    out, lse, idx, _ = _attention(w, t)
            stream.synchronize()
            results[k] = (out, idx, sa.sa_get_status(idx, stream=stream))
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for w, (out, idx, status) in zip(cases, results):
        assert status == 0
        _check(w, out, idx, w.q_host(), w.selected)
