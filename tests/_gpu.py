"""Helpers shared by the GPU tests: put a workload on the device, run the
library through its C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import block_sparse_paged_csr_gb300 as sa
import inputs

TOL_F32 = 1e-4      # f32 arithmetic on the CUDA-core path (row-normalised)
TOL_TC = 2e-2       # tensor-core path (bf16 operands)


def auto_uses_tensor_cores(w) -> bool:
    """Whether SA_PATH_AUTO sends this workload to the tcgen05 kernel (bf16
    operands), as the library itself reports it."""
    return sa.sa_forward_kernel_name(w.tq, w.batch, w.hkv, w.hq, w.head_dim, w.block_size,
                                     w.page_size, w.kv_dtype) == "forward_tc_kernel"


def uses_fused(w) -> bool:
    """Whether sa_attention (SA_PATH_AUTO) takes the fused decode path, which
    writes no partials."""
    return sa.sa_attention_kernel_name(w.cu_seqlens_q, w.num_pages, w.hkv, w.hq, w.head_dim,
                                       w.block_size, w.page_size, w.kv_dtype,
                                       causal=w.causal) == "fused_dec_kernel"


def auto_tol(w) -> float:
    return TOL_TC if auto_uses_tensor_cores(w) else TOL_F32


def device_workload(w: inputs.Workload, dev="cuda", fill_on_device=False):
    """Device tensors of a workload.  Small pools come from the host generator;
    large ones (fill_on_device) from the device fill kernel (same bits)."""
    t = {
        "selected": torch.from_numpy(w.selected).to(dev),
        "cu": torch.from_numpy(w.cu_seqlens_q).to(dev),
        "used": torch.from_numpy(w.used_kv_lens).to(dev) if w.pass_used else None,
        "bt": torch.from_numpy(w.block_tables).to(dev),
    }
    if fill_on_device:
        t["q"], t["k"], t["v"] = inputs.device_tensors(w, dev)
    else:
        t["q"] = torch.from_numpy(w.q_host()).to(dev)
        kh, vh = w.k_host(), w.v_host()
        if w.kv_dtype == "bf16":
            t["k"] = torch.from_numpy(kh.view(np.int16)).to(dev).view(torch.bfloat16)
            t["v"] = torch.from_numpy(vh.view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            t["k"] = torch.from_numpy(kh).to(dev)
            t["v"] = torch.from_numpy(vh).to(dev)
    return t


def run_attention(w, t, split_edges=0, path=sa.PATH_AUTO):
    out, lse, idx, parts = sa.sa_attention(t["q"], t["k"], t["v"], t["selected"],
                                           w.cu_seqlens_q, t["cu"], t["used"], t["bt"], w.hq,
                                           w.hkv, w.head_dim, w.block_size, w.page_size,
                                           w.softmax_scale, w.causal, split_edges=split_edges,
                                           path=path)
    status = sa.sa_get_status(idx)
    assert status == 0, f"device status {sa.sa_status_string(status)}"
    return out, lse, idx, parts


def row_error(got, ref):
    """max over rows of max_d |got - ref| / max(max_d |ref|, 1e-6)."""
    got = np.asarray(got, np.float64).reshape(-1, np.shape(ref)[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, np.shape(ref)[-1])
    den = np.maximum(np.max(np.abs(ref), axis=1), 1e-6)
    return float(np.max(np.max(np.abs(got - ref), axis=1) / den, initial=0.0))


def elementwise_error(got, ref, floor=1e-6):
    """The pages' own metric (gpu.rs, the test comparing the shader with the
    CPU forward): max over elements of |got - ref| / max(|ref|, floor)."""
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


#: (test, quantity, row-normalised error, the pages' element-wise error) of
#: the parity tests, printed at the end of the session (conftest.py).
REPORT = []


def report(test, quantity, got, ref):
    REPORT.append((test, quantity, row_error(got, ref), elementwise_error(got, ref)))


def compare_lse(got, ref, tol):
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), "lse finiteness differs"
    assert np.all(got[~fin] == ref[~fin])
    if fin.any():
        err = np.max(np.abs(got[fin] - ref[fin]) / np.maximum(np.abs(ref[fin]), 1.0))
        assert err <= tol, f"lse error {err:.3e}"


INDEX_KEYS = ("sel_slots", "sel_offsets", "num_sel", "edge_head_base", "edges", "inv", "splits")


def compare_index(got: dict, ref: dict):
    for key in INDEX_KEYS:
        g = np.asarray(got[key], np.int64)
        r = np.asarray(ref[key], np.int64)
        assert g.shape == r.shape, f"{key}: shape {g.shape} vs {r.shape}"
        if not np.array_equal(g, r):
            bad = np.argwhere(g != r)[:5]
            raise AssertionError(f"{key} differs at {bad.tolist()}")
    assert got["n_units"] == ref["n_units"]


def compare_partials(o, m, l, ro, rm, rl, tol):
    o = np.asarray(o, np.float64)
    m = np.asarray(m, np.float64)
    l = np.asarray(l, np.float64)
    dead = rl == 0
    assert np.all(l[dead] == 0) and np.all(np.isneginf(m[dead])) and np.all(o[dead] == 0)
    live = ~dead
    if live.any():
        assert row_error(o[live], ro[live]) <= tol, f"o_partial {row_error(o[live], ro[live])}"
        assert np.max(np.abs(m[live] - rm[live])) <= tol * max(1.0, np.abs(rm[live]).max())
        assert np.max(np.abs(l[live] - rl[live]) / rl[live]) <= tol
