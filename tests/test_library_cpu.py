"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-side checks return the documented status codes before
any device work is enqueued."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sa.h")


@pytest.fixture(scope="module")
def lib():
    from block_sparse_paged_csr_gb300 import _native

    if not os.path.exists(_native.LIB_PATH):
        from block_sparse_paged_csr_gb300 import build

        build.build_library()
    return _native.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    from block_sparse_paged_csr_gb300 import _native

    assert header_functions() == sorted(_native.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    for name in header_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported"


def test_status_strings(lib):
    from block_sparse_paged_csr_gb300 import _native

    for code in _native.STATUS_NAMES:
        assert lib.sa_status_string(code)
    assert b"multiple of Hkv" in lib.sa_status_string(1)
    assert b"sm_103a" in lib.sa_version()


def test_index_sizes_of_the_serving_workloads(lib):
    from block_sparse_paged_csr_gb300 import _native

    s = _native.SaIndexSizes()
    # GQA decode: B=64, 1 query each, Hkv=8, topk=16, max_pages=2048, page 16, block 64
    assert lib.sa_index_query_sizes(64, 8, 16, 64, 2048, 64, 16, ctypes.byref(s)) == 0
    assert (s.msb, s.nbs) == (512, 32768)
    assert s.sel_offsets == 8 * 32769 and s.inv == 64 * 8 * 16 and s.edges == 2 * 8192
    # long-context decode: B=128, Hkv=8, topk=64, max_pages=8192
    assert lib.sa_index_query_sizes(128, 8, 64, 128, 8192, 64, 16, ctypes.byref(s)) == 0
    assert (s.msb, s.nbs) == (2048, 262144)
    # the boundary's workspace-size entry gives the same bytes, and the same errors
    n = ctypes.c_size_t(0)
    assert lib.sa_index_workspace_size(128, 8, 64, 128, 8192, 64, 16, ctypes.byref(n)) == 0
    assert n.value == s.workspace_bytes > 0
    assert lib.sa_index_workspace_size(128, 8, 64, 128, 8192, 64, 16, None) != 0
    assert (lib.sa_index_workspace_size(128, 8, 64, 128, 8192, 40, 16, ctypes.byref(n)) ==
            lib.sa_index_query_sizes(128, 8, 64, 128, 8192, 40, 16, ctypes.byref(s)) != 0)


def _build(lib, **kw):
    from block_sparse_paged_csr_gb300 import _native

    a = dict(selected=None, tq=4, hkv=2, topk=2, cu=np.array([0, 4], np.int64), cu_dev=None,
             batch=1, used=None, max_pages=16, bs=32, ps=16, split=0)
    a.update(kw)
    idx = _native.SaIndex()
    cu = a["cu"]
    return lib.sa_build_index(a["selected"], a["tq"], a["hkv"], a["topk"],
                              cu.ctypes.data_as(ctypes.c_void_p) if cu is not None else None,
                              a["cu_dev"], a["batch"], a["used"], a["max_pages"], a["bs"],
                              a["ps"], a["split"], ctypes.byref(idx), None)


def test_build_index_host_checks(lib):
    names = {v: k for k, v in __import__("block_sparse_paged_csr_gb300._native",
                                         fromlist=["x"]).STATUS_NAMES.items()}
    assert _build(lib, bs=24, ps=16) == names["BLOCK_PAGE"]
    assert _build(lib, bs=0) == names["BLOCK_PAGE"]
    assert _build(lib, tq=0) == names["EMPTY"]
    assert _build(lib, topk=0) == names["EMPTY"]
    assert _build(lib, hkv=0) == names["EMPTY"]
    assert _build(lib, cu=np.array([1, 4], np.int64)) == names["CU_SEQLENS"]
    assert _build(lib, cu=np.array([0, 3, 2, 4], np.int64), batch=3) == names["CU_SEQLENS"]
    assert _build(lib, cu=np.array([0, 3], np.int64)) == names["SHAPE"]
    assert _build(lib, max_pages=2 * 16385) == names["UNSUPPORTED"]
    # everything valid but no device arrays: rejected before any launch
    assert _build(lib) == names["INVALID_ARGUMENT"]


def test_forward_and_combine_host_checks(lib):
    from block_sparse_paged_csr_gb300 import _native

    names = {v: k for k, v in _native.STATUS_NAMES.items()}
    idx = _native.SaIndex(hkv=2, pages_per_block=2, block_size=32, page_size=16, tq=4, topk=2)

    def fwd(hq=4, hkv=2, d=32, bs=32, ps=16, dtype=0, path=0, ptrs=False):
        p = ctypes.c_void_p(16) if ptrs else None
        return lib.sa_forward(p, p, p, 16, dtype, ctypes.byref(idx), p, p, None, hq, hkv, d, bs,
                              ps, 0.1, 0, p, p, p, path, None)

    assert fwd(hq=3) == names["HEAD_COUNT"]
    assert fwd(hkv=0) == names["HEAD_COUNT"]
    assert fwd(bs=24) == names["BLOCK_PAGE"]
    assert fwd(d=0) == names["BLOCK_PAGE"]
    assert fwd(bs=64) == names["SHAPE"]          # index built for another block size
    assert fwd(d=30) == names["UNSUPPORTED"]
    assert fwd(d=512) == names["UNSUPPORTED"]
    assert fwd(dtype=1, d=36) == names["UNSUPPORTED"]
    assert fwd(dtype=7) == names["INVALID_ARGUMENT"]
    assert fwd() == names["INVALID_ARGUMENT"]      # null pointers
    assert lib.sa_combine(ctypes.byref(idx), None, None, None, 3, 32, None, None, None) == \
        names["HEAD_COUNT"]
    assert lib.sa_combine(ctypes.byref(idx), None, None, None, 4, 30, None, None, None) == \
        names["UNSUPPORTED"]


def test_partial_dtype_host_checks(lib):
    """The 16-bit-partial entries: the same checks as their f32 forms, plus
    partial_dtype itself (f32 or bf16 only), all before any launch."""
    from block_sparse_paged_csr_gb300 import _native

    names = {v: k for k, v in _native.STATUS_NAMES.items()}
    idx = _native.SaIndex(hkv=2, pages_per_block=2, block_size=32, page_size=16, tq=4, topk=2)

    def fwd(pdt, hq=4, d=32):
        return lib.sa_forward_ex(None, None, None, 16, 0, ctypes.byref(idx), None, None, None, hq,
                                 2, d, 32, 16, 0.1, 0, pdt, None, None, None, 0, None, None)

    assert fwd(2) == names["INVALID_ARGUMENT"]
    assert fwd(-1) == names["INVALID_ARGUMENT"]
    assert fwd(1, hq=3) == names["HEAD_COUNT"]
    assert fwd(1, d=30) == names["UNSUPPORTED"]
    assert fwd(1) == names["INVALID_ARGUMENT"]       # null pointers
    # a Q scratch that is misaligned, or overlaps q, is refused before any launch
    q = ctypes.c_void_p(4096)
    for scratch in (ctypes.c_void_p(4104), ctypes.c_void_p(4096 + 64)):
        assert lib.sa_forward_ex(q, q, q, 16, 0, ctypes.byref(idx), q, q, None, 4, 2, 32, 32, 16,
                                 0.1, 0, 0, q, q, q, 0, None, scratch) == names["INVALID_ARGUMENT"]
    comb = lib.sa_combine_ex
    assert comb(ctypes.byref(idx), 2, None, None, None, 4, 32, None, None, None) == \
        names["INVALID_ARGUMENT"]
    assert comb(ctypes.byref(idx), 1, None, None, None, 3, 32, None, None, None) == \
        names["HEAD_COUNT"]
    assert comb(ctypes.byref(idx), 1, None, None, None, 4, 32, None, None, None) == \
        names["INVALID_ARGUMENT"]
    host_cu = np.array([0, 4], np.int64)
    assert lib.sa_attention_ex(None, None, None, 16, 0, None, 4, 2, host_cu.ctypes.data, None, 1,
                               None, None, 4, 4, 2, 32, 32, 16, 0.1, 0, 0, ctypes.byref(idx), 5,
                               None, None, None, None, None, 0, None) == names["INVALID_ARGUMENT"]
    assert lib.sa_forward_combine_ex(None, None, None, 16, 0, ctypes.byref(idx), None,
                                     host_cu.ctypes.data, None, None, None, 4, 32, 32, 16, 0.1, 0,
                                     0, 9, None, None, None, None, None, 0, None) == \
        names["INVALID_ARGUMENT"]
    import block_sparse_paged_csr_gb300 as sa
    import torch
    with pytest.raises(ValueError):
        sa._partial_dtype("f16", None)
    with pytest.raises(ValueError):
        sa._partial_dtype("bf16", torch.empty(1, dtype=torch.float32))
    with pytest.raises(TypeError):
        sa._partial_dtype(None, torch.empty(1, dtype=torch.float16))
    assert sa._partial_dtype(None, None) == (torch.float32, 0)
    assert sa._partial_dtype("bf16", None) == (torch.bfloat16, 1)
    assert sa._partial_dtype(None, torch.empty(1, dtype=torch.bfloat16)) == (torch.bfloat16, 1)


def test_forward_kernel_choice(lib):
    """The kernel each serving workload takes under SA_PATH_AUTO and under
    each forced path, and refusals where sa_forward would refuse."""
    import block_sparse_paged_csr_gb300 as sa
    import inputs

    name = sa.sa_forward_kernel_name
    auto = {}
    for wname, builder in inputs.FULL.items():
        w = builder()
        auto[wname] = name(w.tq, w.batch, w.hkv, w.hq, w.head_dim, w.block_size, w.page_size,
                           w.kv_dtype)
    assert auto["gqa_decode"] == "forward_dec_kernel"
    assert auto["long_decode"] == "forward_dec_mma_kernel"
    assert auto["chunked_prefill"] == "forward_tc_kernel"
    assert auto["chunked_prefill_bf16"] == "forward_tc_kernel"
    assert auto["skewed"] == "forward_tc_kernel"
    assert auto["tiny"] == "forward_cc_kernel"      # head_dim 32
    # forced paths on a decode shape (64 sequences, one query each)
    geo = (64, 64, 8, 32, 128, 64, 16)
    assert name(*geo, "f32", sa.PATH_CUDA_CORE) == "forward_dec_kernel"
    assert name(*geo, "bf16", sa.PATH_CUDA_CORE) == "forward_dec_kernel"
    assert name(*geo, "f32", sa.PATH_CUDA_CORE_GENERAL) == "forward_cc_kernel"
    assert name(*geo, "f32", sa.PATH_TENSOR_CORE) == "forward_tc_kernel"
    assert name(*geo, "bf16", sa.PATH_TENSOR_CORE) == "forward_dec_mma_kernel"
    # block 16 is below the decode kernels' two 16-key chunks per block
    assert name(64, 64, 8, 32, 128, 16, 16, "bf16") == "forward_cc_kernel"
    # tensor cores need head_dim 128
    assert name(8192, 4, 8, 64, 64, 128, 64, "f32", sa.PATH_TENSOR_CORE) is None
    assert name(8192, 4, 8, 64, 64, 128, 64, "f32") == "forward_cc_kernel"
    # refusals: head counts, block/page, head_dim beyond the general kernel
    assert name(4, 1, 3, 4, 32, 32, 16) is None
    assert name(4, 1, 2, 4, 32, 32, 24) is None
    assert name(4, 1, 2, 4, 512, 32, 16) is None


def test_attention_kernel_choice(lib):
    """sa_attention's steps 2-3: the fused decode kernel exactly when every
    sequence holds at most one query and the shape is supported."""
    import block_sparse_paged_csr_gb300 as sa
    import inputs

    name = sa.sa_attention_kernel_name
    for wname, fused in (("gqa_decode", True), ("long_decode", True), ("chunked_prefill", False),
                         ("skewed", False), ("tiny", False)):
        w = inputs.FULL[wname]()
        got = name(w.cu_seqlens_q, w.num_pages, w.hkv, w.hq, w.head_dim, w.block_size,
                   w.page_size, w.kv_dtype)
        want = "fused_dec_kernel" if fused else sa.sa_forward_kernel_name(
            w.tq, w.batch, w.hkv, w.hq, w.head_dim, w.block_size, w.page_size, w.kv_dtype)
        assert got == want, (wname, got)
    one = np.array([0, 1, 1, 2, 3], np.int64)          # an empty sequence is allowed
    two = np.array([0, 1, 3, 4], np.int64)             # a sequence with two queries is not
    geo = (1000, 8, 32, 128, 64, 16)
    assert name(one, *geo, "f32") == "fused_dec_kernel"
    assert name(one, *geo, "bf16", sa.PATH_FUSED_DECODE) == "fused_dec_kernel"
    assert name(two, *geo, "f32") == "forward_dec_kernel"
    assert name(two, *geo, "f32", sa.PATH_FUSED_DECODE) is None
    assert name(one, *geo, "f32", sa.PATH_CUDA_CORE) == "forward_dec_kernel"
    # f32 up to 4 q-heads per kv head, bf16 up to 16
    assert name(one, 1000, 8, 64, 128, 64, 16, "f32") == "forward_dec_kernel"
    assert name(one, 1000, 8, 64, 128, 64, 16, "bf16") == "fused_dec_kernel"
    # pages of fewer than 8 keys, or not a power of two, are not fused
    assert name(one, 1000, 8, 32, 128, 64, 4, "f32") != "fused_dec_kernel"
    assert name(one, 1000, 8, 32, 128, 48, 24, "f32") != "fused_dec_kernel"
    # head_dim 128 only
    assert name(one, 1000, 8, 32, 64, 64, 16, "f32") == "forward_cc_kernel"
    # left-aligned causal (causal = 2) leaves the fused path; other modes are refused
    assert name(one, *geo, "f32", causal=1) == "fused_dec_kernel"
    assert name(one, *geo, "f32", causal=2) == "forward_dec_kernel"
    assert name(one, *geo, "f32", sa.PATH_FUSED_DECODE, causal=2) is None
    assert lib.sa_attention_kernel_name(4, 4, one.ctypes.data, 1000, 32, 8, 128, 64, 16, 0, 3,
                                        0) is None
    with pytest.raises(ValueError):
        sa._causal(3)
    assert [sa._causal(c) for c in (False, True, 0, 1, 2)] == [0, 1, 0, 1, 2]


def test_no_alloc_capacity_host_check(lib):
    """sa_build_index_no_alloc refuses, before any device work, exactly the
    problems whose scratch (the formula in sa.h) exceeds its 288 KiB array:
    835 one-query sequences at hkv = 8 pass the size check, 836 do not."""
    from block_sparse_paged_csr_gb300 import _native

    def call(batch):
        cu = np.arange(batch + 1, dtype=np.int64)
        idx = _native.SaIndex()
        return lib.sa_build_index_no_alloc(None, batch, 8, 4, cu.ctypes.data_as(ctypes.c_void_p),
                                           None, batch, None, 40, 64, 16, 0, ctypes.byref(idx),
                                           None)

    assert _native.STATUS_NAMES[call(836)] == "UNSUPPORTED"
    assert _native.STATUS_NAMES[call(835)] != "UNSUPPORTED"
    # a prefill-sized problem (4 x 2048 queries, topk 32, hkv 8, msb 256) does not fit
    cu = np.array([0, 2048, 4096, 6144, 8192], np.int64)
    idx = _native.SaIndex()
    rc = lib.sa_build_index_no_alloc(None, 8192, 8, 32, cu.ctypes.data_as(ctypes.c_void_p), None,
                                     4, None, 512, 128, 64, 0, ctypes.byref(idx), None)
    assert _native.STATUS_NAMES[rc] == "UNSUPPORTED"
