"""KV-outer block-sparse attention over a paged KV cache, for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libsa.so`` (``include/sa.h``).  The
functions carry the same names as the C entry points and do argument
marshalling only: every step of the method runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.

The three steps (crate alice-llm 2.0.0, module sparse_attention):

* :func:`sa_build_index` - CSR index keyed by (kv head, sparse block)
  (``types.rs``, KvOuterIndex);
* :func:`sa_forward` - per-edge partials o, m, l (``forward.rs``,
  kvouter_forward);
* :func:`sa_combine` - log-sum-exp merge per (query, q-head);
* :func:`sa_forward_combine` - steps 2 and 3 on a built index (one fused
  kernel for batches of one query per sequence);
* :func:`sa_attention` - the three on one stream without a host sync.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import _native
from ._native import (DTYPE_BF16, DTYPE_F32, PATH_AUTO, PATH_CUDA_CORE, PATH_CUDA_CORE_GENERAL,
                      PATH_FUSED_DECODE, PATH_TENSOR_CORE, PATH_TENSOR_CORE_TF32, STATUS_NAMES)

__all__ = ["SAError", "Index", "sa_index_query_sizes", "sa_build_index",
           "sa_build_index_no_alloc", "sa_forward", "sa_forward_combine", "sa_forward_kernel_name",
           "sa_attention_kernel_name", "PATH_FUSED_DECODE",
           "sa_combine", "sa_attention", "sa_get_status", "sa_clear_status", "sa_status_string",
           "sa_version", "allocate_index", "PATH_AUTO", "PATH_CUDA_CORE", "PATH_TENSOR_CORE",
           "PATH_TENSOR_CORE_TF32",
           "PATH_CUDA_CORE_GENERAL", "AttentionGraph", "sa_debug_stall", "sa_debug_cta_stats", "STALL_NONE",
           "STALL_INDEX_BARRIER", "STALL_FUSED_COPIES"]

#: sa_debug_stall sites (a test hook: see include/sa.h)
STALL_NONE, STALL_INDEX_BARRIER, STALL_FUSED_COPIES = 0, 1, 2


class SAError(RuntimeError):
    """A non-OK sa_status returned by the library."""

    def __init__(self, code: int, where: str):
        self.code = int(code)
        self.kind = STATUS_NAMES.get(self.code, f"UNKNOWN({code})")
        text = _native.load().sa_status_string(self.code).decode()
        super().__init__(f"{where}: {self.kind} ({text})")


def _causal(causal) -> int:
    """The C ABI's causal mode: 0 none, 1 right-aligned (the pages' rule), 2
    left-aligned (opt-in); booleans map to 0 / 1."""
    if isinstance(causal, (bool, np.bool_)):
        return int(causal)
    c = int(causal)
    if c not in (0, 1, 2):
        raise ValueError(f"causal must be 0, 1 or 2, got {causal!r}")
    return c


def _check(code: int, where: str) -> None:
    if code != _native.SA_OK:
        raise SAError(code, where)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _host_i64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int64)


def _require(t, dtype, name, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def sa_status_string(code: int) -> str:
    return _native.load().sa_status_string(int(code)).decode()


def sa_version() -> str:
    return _native.load().sa_version().decode()


def sa_index_query_sizes(tq, hkv, topk, batch, max_pages, block_size, page_size) -> dict:
    s = _native.SaIndexSizes()
    _check(_native.load().sa_index_query_sizes(tq, hkv, topk, batch, max_pages, block_size,
                                               page_size, ctypes.byref(s)),
           "sa_index_query_sizes")
    return {name: getattr(s, name) for name, _ in s._fields_}


@dataclass
class Index:
    """Device arrays of one KV-outer index plus the C struct that points at them."""

    sel_slots: torch.Tensor
    sel_offsets: torch.Tensor
    num_sel: torch.Tensor
    edge_head_base: torch.Tensor
    edges: torch.Tensor
    inv: torch.Tensor
    splits: torch.Tensor
    totals: torch.Tensor
    workspace: torch.Tensor
    sizes: dict
    c: _native.SaIndex

    @property
    def device(self):
        return self.totals.device

    def to_host(self) -> dict:
        """Copies of the index arrays, shaped and trimmed like the oracle's."""
        c = self.c
        tot = self.totals.cpu().numpy()
        E, S, U = int(tot[0]), int(tot[1]), int(tot[2])
        hkv, nbs, tq, topk = c.hkv, c.nbs, c.tq, c.topk
        return {
            "sel_slots": self.sel_slots[: hkv * nbs].cpu().numpy().reshape(hkv, nbs),
            "sel_offsets": self.sel_offsets.cpu().numpy().reshape(hkv, nbs + 1),
            "num_sel": self.num_sel.cpu().numpy(),
            "edge_head_base": self.edge_head_base.cpu().numpy(),
            "edges": self.edges.view(-1, 2)[:E].cpu().numpy(),
            "inv": self.inv.cpu().numpy().reshape(hkv, tq, topk),
            "splits": self.splits.view(-1, 4)[:S].cpu().numpy(),
            "n_units": U, "status": int(tot[3]),
        }


def allocate_index(tq, hkv, topk, batch, max_pages, block_size, page_size, device) -> Index:
    """Allocate (with torch) every array an index over these sizes needs."""
    s = sa_index_query_sizes(tq, hkv, topk, batch, max_pages, block_size, page_size)
    dev = torch.device(device)
    i32 = dict(dtype=torch.int32, device=dev)
    i64 = dict(dtype=torch.int64, device=dev)
    ws_words = (s["workspace_bytes"] + 255) // 8 + 32
    idx = Index(
        sel_slots=torch.empty(max(s["sel_slots"], 1), **i32),
        sel_offsets=torch.empty(max(s["sel_offsets"], 1), **i32),
        num_sel=torch.empty(max(s["num_sel"], 1), **i32),
        edge_head_base=torch.empty(max(s["edge_head_base"], 1), **i64),
        edges=torch.empty(max(s["edges"], 4), **i32),
        inv=torch.empty(max(s["inv"], 1), **i32),
        splits=torch.empty(max(s["splits"], 4), **i32),
        totals=torch.zeros(max(s["totals"], 4), **i64),
        workspace=torch.empty(ws_words, **i64),
        sizes=s,
        c=_native.SaIndex(),
    )
    c = idx.c
    c.sel_slots = idx.sel_slots.data_ptr()
    c.sel_offsets = idx.sel_offsets.data_ptr()
    c.num_sel = idx.num_sel.data_ptr()
    c.edge_head_base = idx.edge_head_base.data_ptr()
    c.edges = idx.edges.data_ptr()
    c.inv = idx.inv.data_ptr()
    c.splits = idx.splits.data_ptr()
    c.totals = idx.totals.data_ptr()
    base = idx.workspace.data_ptr()
    aligned = (base + 255) & ~255
    c.workspace = aligned
    c.workspace_bytes = idx.workspace.numel() * 8 - (aligned - base)
    return idx


def sa_build_index(selected, cu_seqlens_q_host, cu_seqlens_q, used_kv_lens, max_pages,
                   block_size, page_size, split_edges=0, index: Index | None = None,
                   stream=None) -> Index:
    """Step 1.  ``selected`` [tq, hkv, topk] int32 (device), ``cu_seqlens_q_host``
    the host copy (numpy / CPU tensor) of ``cu_seqlens_q`` [B+1] int64 (device),
    ``used_kv_lens`` [B] int32 (device) or None."""
    _require(selected, torch.int32, "selected")
    dev = selected.device
    tq, hkv, topk = (int(x) for x in selected.shape)
    cu_h = _host_i64(cu_seqlens_q_host)
    _require(cu_seqlens_q, torch.int64, "cu_seqlens_q", dev)
    batch = cu_h.size - 1
    if used_kv_lens is not None:
        _require(used_kv_lens, torch.int32, "used_kv_lens", dev)
    if index is None:
        index = allocate_index(tq, hkv, topk, max(batch, 1), max_pages, block_size, page_size,
                               dev)
    _check(_native.load().sa_build_index(
        _ptr(selected), tq, hkv, topk, cu_h.ctypes.data_as(ctypes.c_void_p), _ptr(cu_seqlens_q),
        batch, _ptr(used_kv_lens), max_pages, block_size, page_size, split_edges,
        ctypes.byref(index.c), _stream(stream, dev)), "sa_build_index")
    return index


def sa_build_index_no_alloc(selected, cu_seqlens_q_host, cu_seqlens_q, used_kv_lens, index: Index,
                            max_pages, block_size, page_size, split_edges=0, stream=None) -> Index:
    """Step 1 with the build's scratch taken from a fixed array inside the
    library instead of ``index.workspace``: for callers that cannot allocate
    device memory at call time.  ``index`` must already hold the output arrays
    (see :func:`allocate_index`).  Calls that overlap on the GPU share that
    array and race; the first call on a device must come before any stream
    capture on it."""
    _require(selected, torch.int32, "selected")
    dev = selected.device
    tq, hkv, topk = (int(x) for x in selected.shape)
    cu_h = _host_i64(cu_seqlens_q_host)
    _require(cu_seqlens_q, torch.int64, "cu_seqlens_q", dev)
    if used_kv_lens is not None:
        _require(used_kv_lens, torch.int32, "used_kv_lens", dev)
    _check(_native.load().sa_build_index_no_alloc(
        _ptr(selected), tq, hkv, topk, cu_h.ctypes.data_as(ctypes.c_void_p), _ptr(cu_seqlens_q),
        cu_h.size - 1, _ptr(used_kv_lens), max_pages, block_size, page_size, split_edges,
        ctypes.byref(index.c), _stream(stream, dev)), "sa_build_index_no_alloc")
    return index


def _kv_dtype(k):
    if k.dtype == torch.float32:
        return DTYPE_F32
    if k.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"k_pages/v_pages must be float32 or bfloat16, got {k.dtype}")


def sa_forward_kernel_name(tq, batch, hkv, hq, head_dim, block_size, page_size, kv_dtype="f32",
                           path=PATH_AUTO):
    """Name of the kernel sa_forward launches for this problem shape, or None
    where sa_forward would refuse it.  Host only."""
    dt = {"f32": DTYPE_F32, "bf16": DTYPE_BF16}[kv_dtype]
    name = _native.load().sa_forward_kernel_name(int(tq), int(batch), hq, hkv, head_dim,
                                                 block_size, page_size, dt, int(path))
    return None if name is None else name.decode()


def sa_attention_kernel_name(cu_seqlens_q_host, num_pages, hkv, hq, head_dim, block_size,
                             page_size, kv_dtype="f32", path=PATH_AUTO, causal=0):
    """The kernel sa_attention runs for steps 2 and 3 ("fused_dec_kernel" on
    the fused decode path), or None where it would refuse the call."""
    cu = _host_i64(cu_seqlens_q_host)
    dt = {"f32": DTYPE_F32, "bf16": DTYPE_BF16}[kv_dtype]
    name = _native.load().sa_attention_kernel_name(
        int(cu[-1]), len(cu) - 1, cu.ctypes.data, int(num_pages), hq, hkv, head_dim, block_size,
        page_size, dt, _causal(causal), int(path))
    return None if name is None else name.decode()


_PARTIAL_DTYPES = {"f32": (torch.float32, 0), "bf16": (torch.bfloat16, 1)}


def _partial_dtype(partial_dtype, o_partial):
    """(torch dtype, sa_dtype code) of the o partials: from ``o_partial`` when
    given (float32 or bfloat16), else ``partial_dtype`` ("f32" default, or
    "bf16": 16-bit o partials, an opt-in the pages do not have)."""
    if o_partial is not None:
        for name, (dt, code) in _PARTIAL_DTYPES.items():
            if o_partial.dtype == dt:
                if partial_dtype not in (None, name):
                    raise ValueError(f"o_partial is {o_partial.dtype}, partial_dtype {partial_dtype}")
                return dt, code
        raise TypeError(f"o_partial must be float32 or bfloat16, got {o_partial.dtype}")
    if partial_dtype is None:
        partial_dtype = "f32"
    if partial_dtype not in _PARTIAL_DTYPES:
        raise ValueError(f"partial_dtype must be 'f32' or 'bf16', got {partial_dtype!r}")
    return _PARTIAL_DTYPES[partial_dtype]


def partial_rows(index: Index, hq: int) -> int:
    """Row capacity of the partial buffers: tq * hkv * topk * qhead."""
    c = index.c
    return max(c.tq * c.hkv * c.topk * (hq // c.hkv), 1)


def sa_forward(q, k_pages, v_pages, index: Index, block_tables, cu_seqlens_q, used_kv_lens, hq,
               hkv, head_dim, block_size, page_size, softmax_scale, causal, o_partial=None,
               m_partial=None, l_partial=None, path=PATH_AUTO, stream=None, partial_dtype=None,
               q_scratch=None):
    """Step 2.  Returns (o_partial, m_partial, l_partial); the first
    totals[0] * qhead rows are valid.  ``partial_dtype="bf16"`` (or a
    bfloat16 ``o_partial``) stores o in bf16; ``q_scratch`` (a tensor of at
    least tq * hq * head_dim * 2 bytes, e.g. the combine's ``out``) lets the
    tensor-core kernel gather Q from a bf16 copy (both: sa_forward_ex)."""
    _require(q, torch.float32, "q")
    dev = q.device
    kvd = _kv_dtype(k_pages)
    _require(k_pages, k_pages.dtype, "k_pages", dev)
    _require(v_pages, k_pages.dtype, "v_pages", dev)
    _require(block_tables, torch.int32, "block_tables", dev)
    _require(cu_seqlens_q, torch.int64, "cu_seqlens_q", dev)
    if used_kv_lens is not None:
        _require(used_kv_lens, torch.int32, "used_kv_lens", dev)
    page_elems = hkv * page_size * head_dim
    num_pages = k_pages.numel() // page_elems if page_elems > 0 else 0
    rows = partial_rows(index, hq) if hkv > 0 and hq % max(hkv, 1) == 0 else 1
    odt, ocode = _partial_dtype(partial_dtype, o_partial)
    if o_partial is None:
        o_partial = torch.empty((rows, head_dim), dtype=odt, device=dev)
    if m_partial is None:
        m_partial = torch.empty(rows, dtype=torch.float32, device=dev)
    if l_partial is None:
        l_partial = torch.empty(rows, dtype=torch.float32, device=dev)
    L = _native.load()
    head = (_ptr(q), _ptr(k_pages), _ptr(v_pages), num_pages, kvd, ctypes.byref(index.c),
            _ptr(block_tables), _ptr(cu_seqlens_q), _ptr(used_kv_lens), hq, hkv, head_dim,
            block_size, page_size, softmax_scale, _causal(causal))
    tail = (_ptr(o_partial), _ptr(m_partial), _ptr(l_partial), path, _stream(stream, dev))
    if q_scratch is not None:
        need = index.c.tq * hq * head_dim * 2
        if q_scratch.device != dev or q_scratch.numel() * q_scratch.element_size() < need:
            raise ValueError(f"q_scratch needs {need} bytes on {dev}")
    if ocode or q_scratch is not None:
        _check(L.sa_forward_ex(*head, ocode, *tail, _ptr(q_scratch)), "sa_forward_ex")
    else:
        _check(L.sa_forward(*head, *tail), "sa_forward")
    return o_partial, m_partial, l_partial


def sa_combine(index: Index, o_partial, m_partial, l_partial, hq, head_dim, out=None, lse=None,
               with_lse=True, stream=None):
    """Step 3.  Returns (out [tq, hq, d], lse [tq, hq] or None).  A bfloat16
    ``o_partial`` is read as 16-bit o partials (sa_combine_ex)."""
    dev = o_partial.device
    tq = index.c.tq
    _, ocode = _partial_dtype(None, o_partial)
    if out is None:
        out = torch.empty((tq, hq, head_dim), dtype=torch.float32, device=dev)
    if lse is None and with_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=dev)
    L = _native.load()
    tail = (_ptr(o_partial), _ptr(m_partial), _ptr(l_partial), hq, head_dim, _ptr(out), _ptr(lse),
            _stream(stream, dev))
    if ocode:
        _check(L.sa_combine_ex(ctypes.byref(index.c), ocode, *tail), "sa_combine_ex")
    else:
        _check(L.sa_combine(ctypes.byref(index.c), *tail), "sa_combine")
    return out, lse


def sa_forward_combine(q, k_pages, v_pages, index: Index, selected, cu_seqlens_q_host,
                       cu_seqlens_q, used_kv_lens, block_tables, hq, head_dim, block_size,
                       page_size, softmax_scale, causal, split_edges=0, partials=None, out=None,
                       lse=None, with_lse=True, path=PATH_AUTO, stream=None, partial_dtype=None):
    """Steps 2 and 3 on a built index (the fused decode kernel where it
    applies).  Returns (out, lse, (o, m, l)).  ``partial_dtype="bf16"`` (or a
    bfloat16 o in ``partials``): 16-bit o partials."""
    _require(q, torch.float32, "q")
    dev = q.device
    kvd = _kv_dtype(k_pages)
    c = index.c
    hkv = c.hkv
    cu_h = _host_i64(cu_seqlens_q_host)
    rows = partial_rows(index, hq) if hkv > 0 and hq % max(hkv, 1) == 0 else 1
    odt, ocode = _partial_dtype(partial_dtype, None if partials is None else partials[0])
    if partials is None:
        partials = (torch.empty((rows, head_dim), dtype=odt, device=dev),
                    torch.empty(rows, dtype=torch.float32, device=dev),
                    torch.empty(rows, dtype=torch.float32, device=dev))
    if out is None:
        out = torch.empty((c.tq, hq, head_dim), dtype=torch.float32, device=dev)
    if lse is None and with_lse:
        lse = torch.empty((c.tq, hq), dtype=torch.float32, device=dev)
    page_elems = hkv * page_size * head_dim
    num_pages = k_pages.numel() // page_elems if page_elems > 0 else 0
    o, m, l = partials
    L = _native.load()
    head = (_ptr(q), _ptr(k_pages), _ptr(v_pages), num_pages, kvd, ctypes.byref(c),
            _ptr(selected), cu_h.ctypes.data_as(ctypes.c_void_p), _ptr(cu_seqlens_q),
            _ptr(used_kv_lens), _ptr(block_tables), hq, head_dim, block_size, page_size,
            softmax_scale, _causal(causal), split_edges)
    tail = (_ptr(o), _ptr(m), _ptr(l), _ptr(out), _ptr(lse), path, _stream(stream, dev))
    if ocode:
        _check(L.sa_forward_combine_ex(*head, ocode, *tail), "sa_forward_combine_ex")
    else:
        _check(L.sa_forward_combine(*head, *tail), "sa_forward_combine")
    return out, lse, partials


def sa_attention(q, k_pages, v_pages, selected, cu_seqlens_q_host, cu_seqlens_q, used_kv_lens,
                 block_tables, hq, hkv, head_dim, block_size, page_size, softmax_scale, causal,
                 split_edges=0, index: Index | None = None, partials=None, out=None, lse=None,
                 with_lse=True, path=PATH_AUTO, stream=None, partial_dtype=None):
    """Steps 1-3 in one call.  Returns (out, lse, index, (o, m, l)).  Pass
    ``index`` / ``partials`` / ``out`` back in to reuse their memory.
    ``partial_dtype="bf16"`` (or a bfloat16 o in ``partials``): 16-bit o
    partials (sa_attention_ex)."""
    _require(q, torch.float32, "q")
    dev = q.device
    kvd = _kv_dtype(k_pages)
    tq, hkv_s, topk = (int(x) for x in selected.shape)
    cu_h = _host_i64(cu_seqlens_q_host)
    batch = cu_h.size - 1
    max_pages = int(block_tables.shape[1])
    if index is None:
        index = allocate_index(tq, hkv_s, topk, max(batch, 1), max_pages, block_size, page_size,
                               dev)
    rows = max(tq * hkv_s * topk * (hq // max(hkv_s, 1)), 1)
    odt, ocode = _partial_dtype(partial_dtype, None if partials is None else partials[0])
    if partials is None:
        partials = (torch.empty((rows, head_dim), dtype=odt, device=dev),
                    torch.empty(rows, dtype=torch.float32, device=dev),
                    torch.empty(rows, dtype=torch.float32, device=dev))
    if out is None:
        out = torch.empty((tq, hq, head_dim), dtype=torch.float32, device=dev)
    if lse is None and with_lse:
        lse = torch.empty((tq, hq), dtype=torch.float32, device=dev)
    page_elems = hkv * page_size * head_dim
    num_pages = k_pages.numel() // page_elems if page_elems > 0 else 0
    o, m, l = partials
    L = _native.load()
    head = (_ptr(q), _ptr(k_pages), _ptr(v_pages), num_pages, kvd, _ptr(selected), tq, topk,
            cu_h.ctypes.data_as(ctypes.c_void_p), _ptr(cu_seqlens_q), batch, _ptr(used_kv_lens),
            _ptr(block_tables), max_pages, hq, hkv, head_dim, block_size, page_size,
            softmax_scale, _causal(causal), split_edges, ctypes.byref(index.c))
    tail = (_ptr(o), _ptr(m), _ptr(l), _ptr(out), _ptr(lse), path, _stream(stream, dev))
    if ocode:
        _check(L.sa_attention_ex(*head, ocode, *tail), "sa_attention_ex")
    else:
        _check(L.sa_attention(*head, *tail), "sa_attention")
    return out, lse, index, partials


class AttentionGraph:
    """Steps 1-3 (sa_attention) captured once into a CUDA graph on fixed
    buffers and replayed: for small decode batches, where the launches of
    the index, forward and combine kernels cost as much as their work.

    Every argument is bound at capture: the device tensors by address (their
    contents may change between replays: new queries, selections, block
    tables, lengths) and the host-side facts the library decides on at call
    time (cu_seqlens_q_host, head counts, sizes, path), which must then stay
    what they were.  ``replay()`` enqueues the graph on the current stream
    and returns (out, lse); status checks go through ``sa_get_status(self.index)``.
    """

    def __init__(self, q, k_pages, v_pages, selected, cu_seqlens_q_host, cu_seqlens_q,
                 used_kv_lens, block_tables, hq, hkv, head_dim, block_size, page_size,
                 softmax_scale, causal, split_edges=0, path=PATH_AUTO, partial_dtype=None):
        args = (q, k_pages, v_pages, selected, cu_seqlens_q_host, cu_seqlens_q, used_kv_lens,
                block_tables, hq, hkv, head_dim, block_size, page_size, softmax_scale, causal)
        kw = dict(split_edges=split_edges, path=path)
        # one eager call first: buffers, library load and kernel attributes
        self.out, self.lse, self.index, self.partials = sa_attention(
            *args, partial_dtype=partial_dtype, **kw)
        torch.cuda.synchronize(q.device)
        status = sa_get_status(self.index)
        if status != 0:
            raise SAError(status, "AttentionGraph (eager call)")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            sa_attention(*args, index=self.index, partials=self.partials, out=self.out,
                         lse=self.lse, **kw)

    def replay(self):
        self.graph.replay()
        return self.out, self.lse


def sa_get_status(index: Index, stream=None) -> int:
    """Synchronise and return the device status code (0 = OK)."""
    return int(_native.load().sa_get_status(ctypes.byref(index.c),
                                            _stream(stream, index.device)))


def sa_clear_status(index: Index, stream=None) -> None:
    _check(_native.load().sa_clear_status(ctypes.byref(index.c), _stream(stream, index.device)),
           "sa_clear_status")


def sa_debug_stall(site: int, spin_limit: int = 0) -> None:
    """Test hook: make the bounded wait at ``site`` run out on every launch
    from now on (STALL_INDEX_BARRIER, STALL_FUSED_COPIES), with ``spin_limit``
    tries per wait (0 = the library default); STALL_NONE restores normal
    operation."""
    _check(_native.load().sa_debug_stall(int(site), int(spin_limit)), "sa_debug_stall")


def sa_debug_cta_stats(stats=None) -> None:
    """Test hook: with ``stats`` (a zeroed int64 CUDA tensor of 3 * n_ctas
    elements) every later tensor-core forward adds each CTA's claimed rows
    and units and writes its busy cycles there; None turns it off."""
    if stats is None:
        _check(_native.load().sa_debug_cta_stats(None, 0), "sa_debug_cta_stats")
        return
    _require(stats, torch.int64, "stats")
    _check(_native.load().sa_debug_cta_stats(_ptr(stats), stats.numel() // 3),
           "sa_debug_cta_stats")
