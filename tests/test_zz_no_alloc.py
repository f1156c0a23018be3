"""sa_build_index_no_alloc against sa_build_index, through the C ABI.

The allocation-free variant serves callers that cannot allocate device memory
when they call (fixed memory pools, memory caps, hosts without a device
allocator): its scratch is an array inside the library.  Checked here:

* two calls in a row, on different inputs, each give exactly the index the
  regular entry point builds with a caller-provided workspace (the second call
  also shows that the shared scratch is cleared between calls);
* the forward entry points run on an index built this way, with the caller's
  workspace field holding garbage or NULL, and match the oracle: the fused
  decode kernel's piece counters and the tensor-core kernel's work counter
  come from the library's array, not from the caller's workspace;
* the capacity stated in sa.h is exact: the largest problem it admits builds
  and matches sa_build_index, one more sequence is refused.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import _gpu
import block_sparse_paged_csr_gb300 as sa
import inputs
import oracle
from block_sparse_paged_csr_gb300 import _native

pytestmark = pytest.mark.gpu

KEYS = ("sel_slots", "sel_offsets", "num_sel", "edge_head_base", "edges", "inv", "splits")
SCRATCH_BYTES = 288 * 1024


def _c_build(fn_name, w, t, index, split):
    lib = _native.load()
    cu_h = np.ascontiguousarray(w.cu_seqlens_q, dtype=np.int64)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    fn = getattr(lib, fn_name)
    used = t.get("used")
    return fn(ctypes.c_void_p(t["selected"].data_ptr()), w.tq, w.hkv, w.topk,
              cu_h.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(t["cu"].data_ptr()),
              w.batch, None if used is None else ctypes.c_void_p(used.data_ptr()), w.max_pages,
              w.block_size, w.page_size, split, ctypes.byref(index.c), stream)


def _alloc(w):
    return sa.allocate_index(w.tq, w.hkv, w.topk, w.batch, w.max_pages, w.block_size,
                             w.page_size, "cuda")


@pytest.mark.parametrize("first,second", [("skewed", "gqa_decode"),
                                          ("chunked_prefill", "long_decode")])
def test_no_alloc_matches_workspace_build_twice(first, second):
    for name, split in ((first, 3), (second, 0)):
        w = inputs.small(name, seed=5)
        t = _gpu.device_workload(w)
        ref, got = _alloc(w), _alloc(w)
        ws_before = got.c.workspace
        assert _c_build("sa_build_index", w, t, ref, split) == 0
        assert _c_build("sa_build_index_no_alloc", w, t, got, split) == 0
        assert sa.sa_get_status(ref) == 0 and sa.sa_get_status(got) == 0
        assert got.c.workspace == ws_before, "the caller's workspace field is left as it was"
        assert got.c.flags == 1 and ref.c.flags == 0
        a, b = ref.to_host(), got.to_host()
        for key in KEYS:
            assert np.array_equal(a[key], b[key]), f"{name}: {key} differs"
        assert a["n_units"] == b["n_units"]


def _oracle(w):
    return oracle.attention(w.q_host(), w.k_host(), w.v_host(), w.selected, w.block_tables,
                            w.cu_seqlens_q, w.used, w.hq, w.head_dim, w.block_size, w.page_size,
                            w.softmax_scale, w.causal)


@pytest.mark.parametrize("workspace", ["garbage", "null"])
@pytest.mark.parametrize("name", ["gqa_decode", "long_decode", "skewed", "chunked_prefill"])
def test_forward_on_a_no_alloc_index(name, workspace):
    """sa_forward_combine (the fused decode kernel on the decode shapes, the
    tensor-core forward + combine on the others) and sa_forward + sa_combine
    on an index built without a workspace, against the oracle."""
    w = inputs.small(name, seed=7)
    t = _gpu.device_workload(w)
    index = _alloc(w)
    if workspace == "garbage":
        index.workspace.fill_(-1)          # every byte 0xFF
    else:
        index.c.workspace = None
        index.c.workspace_bytes = 0
    assert _c_build("sa_build_index_no_alloc", w, t, index, 0) == 0
    ref_out, ref_lse, _, _ = _oracle(w)
    tol = _gpu.auto_tol(w)
    for _ in range(2):                     # the fused kernel leaves its counters at zero
        out, lse, _ = sa.sa_forward_combine(t["q"], t["k"], t["v"], index, t["selected"],
                                            w.cu_seqlens_q, t["cu"], t["used"], t["bt"], w.hq,
                                            w.head_dim, w.block_size, w.page_size,
                                            w.softmax_scale, w.causal)
        assert sa.sa_get_status(index) == 0
        assert _gpu.row_error(out.cpu().numpy(), ref_out) <= tol
        _gpu.compare_lse(lse.cpu().numpy(), ref_lse, tol)
    o, m, l = sa.sa_forward(t["q"], t["k"], t["v"], index, t["bt"], t["cu"], t["used"], w.hq,
                            w.hkv, w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                            w.causal)
    out, lse = sa.sa_combine(index, o, m, l, w.hq, w.head_dim)
    assert sa.sa_get_status(index) == 0
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= _gpu.auto_tol(w)
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, _gpu.auto_tol(w))


def _scratch_bytes(hkv, batch, tq, multi_chunks, msb):
    """The capacity formula of sa.h (sa_build_index_no_alloc)."""
    up = lambda x: (x + 255) // 256 * 256
    s = hkv * batch
    a = up(256 + 4 * s)
    b = up(a + 4 * hkv * tq)
    c = up(b + 12 * s)
    d = up(c + 24 * (s + 1))
    return up(d + 4 * hkv * multi_chunks * msb)


def _decode_batch(batch, seed=3):
    return inputs.gqa_decode(seed, batch=batch, kv_min=300, kv_max=600, hq=8, hkv=8,
                             head_dim=32, topk=4)


def _index_inputs(w):
    """Only what the index build reads (no K/V pool)."""
    return {"selected": torch.from_numpy(w.selected).cuda(),
            "cu": torch.from_numpy(w.cu_seqlens_q).cuda(),
            "used": torch.from_numpy(w.used_kv_lens).cuda()}


def test_no_alloc_capacity_boundary():
    """The largest batch the formula admits builds (and equals the workspace
    build); one more sequence is refused with SA_ERR_UNSUPPORTED."""
    n = 1
    while _scratch_bytes(8, n + 1, n + 1, 0, 16) <= SCRATCH_BYTES:
        n += 1
    assert _scratch_bytes(8, n, n, 0, 16) <= SCRATCH_BYTES < _scratch_bytes(8, n + 1, n + 1, 0, 16)
    w = _decode_batch(n)
    assert w.msb <= 16 and w.hkv == 8 and w.tq == n
    t = _index_inputs(w)
    ref, got = _alloc(w), _alloc(w)
    assert _c_build("sa_build_index", w, t, ref, 0) == 0
    assert _c_build("sa_build_index_no_alloc", w, t, got, 0) == 0
    assert sa.sa_get_status(ref) == 0 and sa.sa_get_status(got) == 0
    a, b = ref.to_host(), got.to_host()
    for key in KEYS:
        assert np.array_equal(a[key], b[key]), f"{key} differs at the capacity limit"
    w2 = _decode_batch(n + 1)
    t2 = _index_inputs(w2)
    over = _alloc(w2)
    rc = _c_build("sa_build_index_no_alloc", w2, t2, over, 0)
    assert _native.STATUS_NAMES[rc] == "UNSUPPORTED"


def test_no_alloc_rejects_too_many_segments():
    w = inputs.small("gqa_decode", seed=5)
    idx = _native.SaIndex()
    cu = np.zeros(40001, np.int64)
    lib = _native.load()
    rc = lib.sa_build_index_no_alloc(None, 1, 8, 1, cu.ctypes.data_as(ctypes.c_void_p), None,
                                     40000, None, w.max_pages, w.block_size, w.page_size, 0,
                                     ctypes.byref(idx), None)
    assert _native.STATUS_NAMES[rc] == "UNSUPPORTED"
