"""sa_build_index_no_alloc against sa_build_index, through the C ABI.

The allocation-free variant serves callers that cannot allocate device memory
when they call (fixed memory pools, memory caps, hosts without a device
allocator): its scratch is an array inside the library.  Two calls in a row,
on different inputs, must each give exactly the index the regular entry point
builds with a caller-provided workspace; the second call also shows that the
shared scratch is cleared between calls.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_paged_csr_gb300 as sa
import inputs
from block_sparse_paged_csr_gb300 import _native

pytestmark = pytest.mark.gpu

KEYS = ("sel_slots", "sel_offsets", "num_sel", "edge_head_base", "edges", "inv", "splits")


def _c_build(fn_name, w, t, index, split):
    lib = _native.load()
    cu_h = np.ascontiguousarray(w.cu_seqlens_q, dtype=np.int64)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    fn = getattr(lib, fn_name)
    return fn(ctypes.c_void_p(t["sel"].data_ptr()), w.tq, w.hkv, w.topk,
              cu_h.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(t["cu"].data_ptr()),
              w.batch, ctypes.c_void_p(t["used"].data_ptr()), w.max_pages, w.block_size,
              w.page_size, split, ctypes.byref(index.c), stream)


def _tensors(w):
    return {"sel": torch.from_numpy(w.selected).cuda(),
            "cu": torch.from_numpy(w.cu_seqlens_q).cuda(),
            "used": torch.from_numpy(w.used_kv_lens).cuda()}


@pytest.mark.parametrize("first,second", [("skewed", "gqa_decode"),
                                          ("chunked_prefill", "long_decode")])
def test_no_alloc_matches_workspace_build_twice(first, second):
    for name, split in ((first, 3), (second, 0)):
        w = inputs.small(name, seed=5)
        t = _tensors(w)
        ref = sa.allocate_index(w.tq, w.hkv, w.topk, w.batch, w.max_pages, w.block_size,
                                w.page_size, "cuda")
        got = sa.allocate_index(w.tq, w.hkv, w.topk, w.batch, w.max_pages, w.block_size,
                                w.page_size, "cuda")
        ws_before = got.c.workspace
        assert _c_build("sa_build_index", w, t, ref, split) == 0
        assert _c_build("sa_build_index_no_alloc", w, t, got, split) == 0
        assert sa.sa_get_status(ref) == 0 and sa.sa_get_status(got) == 0
        assert got.c.workspace == ws_before, "the caller's workspace field is left as it was"
        a, b = ref.to_host(), got.to_host()
        for key in KEYS:
            assert np.array_equal(a[key], b[key]), f"{name}: {key} differs"
        assert a["n_units"] == b["n_units"]


def test_no_alloc_rejects_too_many_segments():
    w = inputs.small("gqa_decode", seed=5)
    idx = _native.SaIndex()
    cu = np.zeros(40001, np.int64)
    lib = _native.load()
    rc = lib.sa_build_index_no_alloc(None, 1, 8, 1, cu.ctypes.data_as(ctypes.c_void_p), None,
                                     40000, None, w.max_pages, w.block_size, w.page_size, 0,
                                     ctypes.byref(idx), None)
    assert _native.STATUS_NAMES[rc] == "UNSUPPORTED"
