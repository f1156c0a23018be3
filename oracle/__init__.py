"""Oracle for KV-outer block-sparse paged attention (test infrastructure).

A plain CPU statement, in double precision, of the three steps the crate
alice-llm 2.0.0 (module ``sparse_attention``) defines: the KV-outer CSR index
(``types.rs``, ``KvOuterIndex``), the per-edge partials (``forward.rs``,
``kvouter_forward`` / ``process_work_unit``) and the log-sum-exp combine
(``forward.rs`` module doc), plus an independent query-outer attention used as
a cross-check.  The arithmetic lives in ``sa_oracle.c``; this module compiles it
with gcc and marshals numpy arrays.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

ERROR_NAMES = {
    0: "OK",
    1: "HEAD_COUNT",
    2: "BLOCK_PAGE",
    3: "CU_SEQLENS",
    4: "SHAPE",
    5: "SELECTED_RANGE",
    6: "HEAD_DIM",
    7: "EMPTY",
}


class OracleError(RuntimeError):
    """An error kind of the pages' error enum, raised by the oracle."""

    def __init__(self, code: int):
        self.code = code
        self.kind = ERROR_NAMES.get(code, f"UNKNOWN({code})")
        super().__init__(self.kind)


_lock = threading.Lock()
_lib = None


def compile_library(source: str = _SRC, out_path: str = _LIB_PATH) -> str:
    """Compile the oracle's C source into a shared library with gcc."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, source, "-lm"],
        check=True,
    )
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_library()
    return _LIB_PATH


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_validate_cu_seqlens.argtypes = [p, i64]
    lib.orc_validate_cu_seqlens.restype = ctypes.c_int
    lib.orc_batch_of.argtypes = [p, i64, i64]
    lib.orc_batch_of.restype = i64
    lib.orc_selection_get.argtypes = [p, i64, i64, i64, i64, i64]
    lib.orc_selection_get.restype = ctypes.c_int32
    lib.orc_index_geometry.argtypes = [i64] * 7 + [p, p]
    lib.orc_index_geometry.restype = None
    lib.orc_build_index.argtypes = [p, i64, i64, i64, p, i64, p, i64, i64, i64, i64] + [p] * 8
    lib.orc_build_index.restype = ctypes.c_int
    lib.orc_forward.argtypes = ([p, p, p, ctypes.c_int, i64, p, p, p, p, p, i64, i64, p, i64,
                                 p, i64, p, i64, i64, i64, i64, i64, ctypes.c_float,
                                 ctypes.c_int, p, p, p])
    lib.orc_forward.restype = ctypes.c_int
    lib.orc_round_bf16.argtypes = [ctypes.c_double]
    lib.orc_round_bf16.restype = ctypes.c_double
    lib.orc_round_bf16_array.argtypes = [p, i64, p]
    lib.orc_round_bf16_array.restype = None
    lib.orc_combine.argtypes = [p, p, i64, i64, i64, i64, i64, p, p, p, p, p]
    lib.orc_combine.restype = None
    lib.orc_direct.argtypes = ([p, p, p, ctypes.c_int, i64, p, i64, i64, i64, p, i64, p, p,
                                i64, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, p, i64,
                                p, p])
    lib.orc_direct.restype = ctypes.c_int
    return lib


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle shared library from an explicit path (used by tests that
    compile a deliberately altered copy of the source)."""
    return _declare(ctypes.CDLL(path))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def causal_mode(causal) -> int:
    """0 (none), 1 (right-aligned, the code's rule) or 2 (left-aligned, the
    doc's reading for unknown KV lengths); booleans map to 0 / 1."""
    if isinstance(causal, (bool, np.bool_)):
        return int(causal)
    c = int(causal)
    if c not in (0, 1, 2):
        raise ValueError(f"causal must be 0, 1 or 2, got {causal!r}")
    return c


def _check(code: int):
    if code != 0:
        raise OracleError(code)


# --------------------------------------------------------------------------- types


def validate_cu_seqlens(prefix, _lib=None) -> str:
    """CuSeqlensQ::new rules; returns the error kind name ("OK" if valid)."""
    L = _lib or lib()
    a = _c(prefix, np.int64)
    if a.size == 0:
        a = np.zeros(1, np.int64)
        return ERROR_NAMES[L.orc_validate_cu_seqlens(_ptr(a), 0)]
    return ERROR_NAMES[L.orc_validate_cu_seqlens(_ptr(a), a.size)]


def batch_of(prefix, query: int, _lib=None) -> int:
    """CuSeqlensQ::batch_of."""
    L = _lib or lib()
    a = _c(prefix, np.int64)
    return int(L.orc_batch_of(_ptr(a), a.size, query))


def selection_get(selected_flat, hkv: int, topk: int, i: int, h: int, r: int, _lib=None) -> int:
    """SparseSelection::get on a flat row-major buffer."""
    L = _lib or lib()
    a = _c(selected_flat, np.int32)
    return int(L.orc_selection_get(_ptr(a), hkv, topk, i, h, r))


def geometry(tq, hkv, topk, batch, max_pages, block_size, page_size, _lib=None):
    L = _lib or lib()
    msb = ctypes.c_int64()
    nbs = ctypes.c_int64()
    L.orc_index_geometry(tq, hkv, topk, batch, max_pages, block_size, page_size,
                         ctypes.byref(msb), ctypes.byref(nbs))
    return msb.value, nbs.value


# --------------------------------------------------------------------------- step 1


def build_index(selected, cu_seqlens_q, used_kv_lens, max_pages, block_size, page_size,
                split_edges: int = 0, _lib=None) -> dict:
    """KvOuterIndex of ``selected[tq, hkv, topk]`` (int32, -1 = padding).

    Returns a dict of numpy arrays: sel_slots [hkv, nbs], sel_offsets
    [hkv, nbs+1], num_sel [hkv], edges [E, 2], edge_head_base [hkv+1],
    inv [hkv, tq, topk], splits [S, 4] (head, compact slot, edge start, edge
    end), plus the scalars tq, hkv, topk, batch, msb, nbs, ppb, n_units.
    Raises OracleError for the pages' error kinds.
    """
    L = _lib or lib()
    sel = _c(selected, np.int32)
    tq, hkv, topk = (int(x) for x in sel.shape)
    cu = _c(cu_seqlens_q, np.int64)
    batch = cu.size - 1
    used = _c(used_kv_lens, np.int32)
    if block_size <= 0 or page_size <= 0 or block_size % page_size:
        raise OracleError(2)
    msb, nbs = geometry(tq, hkv, topk, batch, max_pages, block_size, page_size, _lib=L)
    n = max(tq * hkv * topk, 1)
    sel_slots = np.empty(max(hkv * nbs, 1), np.int32)
    sel_offsets = np.empty(max(hkv * (nbs + 1), 1), np.int32)
    num_sel = np.empty(max(hkv, 1), np.int32)
    edges = np.empty((n, 2), np.int32)
    ehb = np.empty(hkv + 1, np.int64)
    inv = np.empty(n, np.int32)
    splits = np.empty((n, 4), np.int64)
    totals = np.zeros(3, np.int64)
    if batch < 0:
        raise OracleError(3)
    code = L.orc_build_index(_ptr(sel), tq, hkv, topk, _ptr(cu), batch, _ptr(used), max_pages,
                             block_size, page_size, split_edges, _ptr(sel_slots),
                             _ptr(sel_offsets), _ptr(num_sel), _ptr(edges), _ptr(ehb),
                             _ptr(inv), _ptr(splits), _ptr(totals))
    _check(code)
    E, S, U = (int(x) for x in totals)
    return {
        "sel_slots": sel_slots[: hkv * nbs].reshape(hkv, nbs),
        "sel_offsets": sel_offsets[: hkv * (nbs + 1)].reshape(hkv, nbs + 1),
        "num_sel": num_sel[:hkv].copy(),
        "edges": edges[:E].copy(),
        "edge_head_base": ehb,
        "inv": inv[: hkv * tq * topk].reshape(hkv, tq, topk),
        "splits": splits[:S].copy(),
        "tq": tq, "hkv": hkv, "topk": topk, "batch": batch, "msb": msb, "nbs": nbs,
        "ppb": block_size // page_size, "n_units": U, "max_pages": max_pages,
        "block_size": block_size, "page_size": page_size,
    }


# --------------------------------------------------------------------------- step 2


def _kv(pages):
    """(array, is_bf16): bf16 pools are passed as their uint16 bit patterns."""
    a = np.ascontiguousarray(pages)
    if a.dtype == np.uint16:
        return a, 1
    return np.ascontiguousarray(a, dtype=np.float32), 0


def round_bf16(x, _lib=None):
    """Each value rounded to the nearest bfloat16 (ties to even), as float64."""
    L = _lib or lib()
    a = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(a)
    if a.size:
        L.orc_round_bf16_array(_ptr(a), a.size, _ptr(y))
    return y


def forward(q, k_pages, v_pages, index: dict, block_tables, cu_seqlens_q, used_kv_lens,
            hq: int, head_dim: int, softmax_scale: float, causal: bool, partial_dtype="f32",
            _lib=None):
    """Partials (o [E*qhead, d], m [E*qhead], l [E*qhead]) in float64;
    ``partial_dtype="bf16"``: o rounded to bfloat16 (the opt-in 16-bit o
    partials; m and l unchanged)."""
    assert partial_dtype in ("f32", "bf16")
    L = _lib or lib()
    qa = _c(q, np.float32)
    k, kb = _kv(k_pages)
    v, vb = _kv(v_pages)
    assert kb == vb
    hkv = index["hkv"]
    page_size = index["page_size"]
    block_size = index["block_size"]
    num_pages = k.size // (hkv * page_size * head_dim)
    qhead = hq // hkv if hkv and hq % hkv == 0 else 1
    E = index["edges"].shape[0]
    rows = max(E * qhead, 1)
    o = np.zeros((rows, head_dim), np.float64)
    m = np.zeros(rows, np.float64)
    l = np.zeros(rows, np.float64)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    used = _c(used_kv_lens, np.int32)
    code = L.orc_forward(_ptr(qa), _ptr(k), _ptr(v), kb, num_pages,
                         _ptr(_c(index["sel_slots"], np.int32)),
                         _ptr(_c(index["sel_offsets"], np.int32)),
                         _ptr(_c(index["num_sel"], np.int32)),
                         _ptr(_c(index["edges"], np.int32)),
                         _ptr(_c(index["edge_head_base"], np.int64)),
                         index["nbs"], index["msb"], _ptr(bt), index["max_pages"], _ptr(cu),
                         cu.size - 1, _ptr(used), hq, hkv, head_dim, block_size, page_size,
                         softmax_scale, causal_mode(causal), _ptr(o), _ptr(m), _ptr(l))
    _check(code)
    o = o[: E * qhead]
    if partial_dtype == "bf16":
        o = round_bf16(o, _lib=L)
    return o, m[: E * qhead], l[: E * qhead]


# --------------------------------------------------------------------------- step 3


def combine(index: dict, qhead: int, head_dim: int, o, m, l, _lib=None):
    """Log-sum-exp merge: (out [tq, hq, d], lse [tq, hq]) in float64."""
    L = _lib or lib()
    tq, hkv, topk = index["tq"], index["hkv"], index["topk"]
    out = np.zeros((tq, hkv * qhead, head_dim), np.float64)
    lse = np.zeros((tq, hkv * qhead), np.float64)
    o = _c(o, np.float64)
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    if o.size == 0:
        o, m, l = np.zeros(head_dim), np.zeros(1), np.zeros(1)
    L.orc_combine(_ptr(_c(index["inv"], np.int32)), _ptr(_c(index["edge_head_base"], np.int64)),
                  tq, hkv, topk, qhead, head_dim, _ptr(o), _ptr(m), _ptr(l), _ptr(out),
                  _ptr(lse))
    return out, lse


def attention(q, k_pages, v_pages, selected, block_tables, cu_seqlens_q, used_kv_lens,
              hq, head_dim, block_size, page_size, softmax_scale, causal, split_edges=0,
              partial_dtype="f32", _lib=None):
    """Steps 1-3 in sequence: (out, lse, index, (o, m, l))."""
    bt = np.asarray(block_tables)
    idx = build_index(selected, cu_seqlens_q, used_kv_lens, bt.shape[1], block_size,
                      page_size, split_edges, _lib=_lib)
    qhead = hq // idx["hkv"]
    o, m, l = forward(q, k_pages, v_pages, idx, bt, cu_seqlens_q, used_kv_lens, hq,
                      head_dim, softmax_scale, causal, partial_dtype=partial_dtype, _lib=_lib)
    out, lse = combine(idx, qhead, head_dim, o, m, l, _lib=_lib)
    return out, lse, idx, (o, m, l)


# --------------------------------------------------------------------------- cross-check


def direct(q, k_pages, v_pages, selected, block_tables, cu_seqlens_q, used_kv_lens,
           hq, head_dim, block_size, page_size, softmax_scale, causal, rows=None, _lib=None):
    """Query-outer attention over the selection.  ``rows``: optional [n, 2]
    array of (query, q-head); returns (out [n, d], lse [n]) or, when rows is
    None, (out [tq, hq, d], lse [tq, hq])."""
    L = _lib or lib()
    qa = _c(q, np.float32)
    k, kb = _kv(k_pages)
    v, vb = _kv(v_pages)
    assert kb == vb
    sel = _c(selected, np.int32)
    tq, hkv, topk = (int(x) for x in sel.shape)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int64)
    used = _c(used_kv_lens, np.int32)
    num_pages = k.size // (hkv * page_size * head_dim)
    rws = None if rows is None else _c(rows, np.int64).reshape(-1, 2)
    n = tq * hq if rws is None else rws.shape[0]
    out = np.zeros((max(n, 1), head_dim), np.float64)
    lse = np.zeros(max(n, 1), np.float64)
    code = L.orc_direct(_ptr(qa), _ptr(k), _ptr(v), kb, num_pages, _ptr(sel), tq, hkv, topk,
                        _ptr(cu), cu.size - 1, _ptr(used), _ptr(bt), bt.shape[1], hq, head_dim,
                        block_size, page_size, softmax_scale, causal_mode(causal), _ptr(rws),
                        0 if rws is None else n, _ptr(out), _ptr(lse))
    _check(code)
    if rws is None:
        return out[:n].reshape(tq, hq, head_dim), lse[:n].reshape(tq, hq)
    return out[:n], lse[:n]
