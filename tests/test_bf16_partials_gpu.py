"""The opt-in 16-bit o partials (sa_forward_ex / sa_combine_ex /
sa_attention_ex with SA_DTYPE_BF16) against the oracle's reading of them:
every o value rounded to the nearest bfloat16 before the combine, m and l in
full precision.  Every forward kernel, the fused decode path (whose piece
scratch then holds bf16 o rows), the separate steps, and the full-size
prefill workload on sampled rows.  Tolerance: the bf16 one (2e-2,
row-normalised) throughout."""
import numpy as np
import pytest
import torch

import _gpu
import block_sparse_paged_csr_gb300 as sa
import inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = _gpu.TOL_TC

SMALL = ["tiny", "gqa_decode", "chunked_prefill", "chunked_prefill_bf16", "skewed",
         "long_decode"]
PATHS = {"auto": sa.PATH_AUTO, "cuda_core": sa.PATH_CUDA_CORE,
         "cuda_core_general": sa.PATH_CUDA_CORE_GENERAL, "tensor_core": sa.PATH_TENSOR_CORE}


def _oracle(w, split, partial_dtype):
    return oracle.attention(w.q_host(), w.k_host(), w.v_host(), w.selected, w.block_tables,
                            w.cu_seqlens_q, w.used, w.hq, w.head_dim, w.block_size, w.page_size,
                            w.softmax_scale, w.causal, split_edges=split,
                            partial_dtype=partial_dtype)


def _attention_bf16(w, t, split, path):
    out, lse, idx, parts = sa.sa_attention(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q,
                                           t["cu"], t["used"], t["bt"], w.hq, w.hkv, w.head_dim,
                                           w.block_size, w.page_size, w.softmax_scale, w.causal,
                                           split_edges=split, path=path, partial_dtype="bf16")
    assert sa.sa_get_status(idx) == 0
    return out, lse, idx, parts


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("path", list(PATHS), ids=list(PATHS))
@pytest.mark.parametrize("name", SMALL)
def test_bf16_partials_each_kernel(name, path, split):
    w = inputs.small(name, seed=4)
    if path == "tensor_core" and sa.sa_forward_kernel_name(
            w.tq, w.batch, w.hkv, w.hq, w.head_dim, w.block_size, w.page_size, w.kv_dtype,
            sa.PATH_TENSOR_CORE) is None:
        pytest.skip("no tensor-core kernel for this shape")
    t = _gpu.device_workload(w)
    out, lse, idx, (o, m, l) = _attention_bf16(w, t, split, PATHS[path])
    assert o.dtype == torch.bfloat16
    ref_out, ref_lse, ref_idx, (ro, rm, rl) = _oracle(w, split, "bf16")
    _gpu.compare_index(idx.to_host(), ref_idx)
    if not (path == "auto" and _gpu.uses_fused(w)):
        rows = ref_idx["edges"].shape[0] * w.qhead
        _gpu.compare_partials(o[:rows].float().cpu().numpy(), m[:rows].cpu().numpy(),
                              l[:rows].cpu().numpy(), ro, rm, rl, TOL)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= TOL
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, TOL)


@pytest.mark.parametrize("path", ["cuda_core", "tensor_core"])
def test_bf16_partials_are_the_rounded_f32_partials(path):
    """On one kernel the bf16 o rows are the f32 rows rounded to nearest
    even (the same arithmetic, only the store differs): bit-exact."""
    w = inputs.small("chunked_prefill", seed=6)
    t = _gpu.device_workload(w)
    _, _, idx, (o32, m32, l32) = _gpu.run_attention(w, t, split_edges=3, path=PATHS[path])
    _, _, idx16, (o16, m16, l16) = _attention_bf16(w, t, 3, PATHS[path])
    rows = int(idx.to_host()["edges"].shape[0]) * w.qhead
    assert torch.equal(o32[:rows].to(torch.bfloat16), o16[:rows])
    assert torch.equal(m32[:rows], m16[:rows]) and torch.equal(l32[:rows], l16[:rows])


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("split", [0, 1, 5])
def test_bf16_partials_fused_decode(dt, split):
    """The fused decode path with 16-bit scratch: pieces of a (query, kv
    head) merge through bf16 o rows (18 pairs on the SMs: every split cuts
    pairs into pieces; split 1 gives every rank its own piece).  The
    rounding falls on pieces, not edges, so the reference is the oracle's
    f32-partial output."""
    qhead = 4 if dt == "f32" else 8
    w = inputs.gqa_decode(seed=31, batch=9, kv_min=900, kv_max=2100, hkv=2, hq=2 * qhead,
                          head_dim=128, page_size=16, block_size=64, topk=6, kv_dtype=dt)
    assert _gpu.uses_fused(w)
    t = _gpu.device_workload(w)
    out, lse, idx, _ = _attention_bf16(w, t, split, sa.PATH_AUTO)
    ref_out, ref_lse, ref_idx, _ = _oracle(w, split, "f32")
    _gpu.compare_index(idx.to_host(), ref_idx)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= TOL
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, TOL)


@pytest.mark.parametrize("head_dim", [20, 36])
def test_bf16_partials_head_dim_not_multiple_of_8(head_dim):
    """The general f32 forward and the combine's 8-byte bf16 loads (head_dim
    a multiple of 4 but not of 8)."""
    w = inputs.chunked_prefill(seed=head_dim, batch=2, qo_len=5, kv_len=300, hq=4, hkv=2,
                               head_dim=head_dim, page_size=16, block_size=32, topk=3)
    t = _gpu.device_workload(w)
    out, lse, idx, (o, m, l) = _attention_bf16(w, t, 2, sa.PATH_AUTO)
    ref_out, ref_lse, ref_idx, (ro, rm, rl) = _oracle(w, 2, "bf16")
    _gpu.compare_index(idx.to_host(), ref_idx)
    rows = ref_idx["edges"].shape[0] * w.qhead
    _gpu.compare_partials(o[:rows].float().cpu().numpy(), m[:rows].cpu().numpy(),
                          l[:rows].cpu().numpy(), ro, rm, rl, TOL)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= TOL
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, TOL)


def test_bf16_partials_separate_steps_match_attention():
    w = inputs.small("skewed", seed=8)
    t = _gpu.device_workload(w)
    out, lse, idx, _ = _attention_bf16(w, t, 0, sa.PATH_AUTO)
    idx2 = sa.sa_build_index(t["selected"], w.cu_seqlens_q, t["cu"], t["used"], w.max_pages,
                             w.block_size, w.page_size)
    o, m, l = sa.sa_forward(t["q"], t["k"], t["v"], idx2, t["bt"], t["cu"], t["used"], w.hq,
                            w.hkv, w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                            w.causal, partial_dtype="bf16")
    assert o.dtype == torch.bfloat16
    out2, lse2 = sa.sa_combine(idx2, o, m, l, w.hq, w.head_dim)
    assert sa.sa_get_status(idx2) == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("name", ["chunked_prefill", "chunked_prefill_bf16"])
def test_bf16_partials_full_size_prefill(name):
    """The prefill workload at full size (the launch the benchmark's
    16-bit-partial option times): outputs on sampled rows against the
    oracle's query-outer attention."""
    w = inputs.FULL[name](0)
    t = _gpu.device_workload(w, fill_on_device=True)
    out, lse, idx, _ = _attention_bf16(w, t, 16, sa.PATH_AUTO)
    rng = np.random.default_rng(12)
    queries = np.unique(rng.choice(w.tq, size=12, replace=False))
    k, v, bt, _ = w.compact_pool(queries)
    rows = np.array([(i, hq) for i in queries for hq in rng.choice(w.hq, 4, replace=False)])
    ref, ref_lse = oracle.direct(w.q_host(), k, v, w.selected, bt, w.cu_seqlens_q, w.used, w.hq,
                                 w.head_dim, w.block_size, w.page_size, w.softmax_scale, w.causal,
                                 rows=rows)
    assert _gpu.row_error(out[rows[:, 0], rows[:, 1]].cpu().numpy(), ref) <= TOL
    _gpu.compare_lse(lse[rows[:, 0], rows[:, 1]].cpu().numpy(), ref_lse, TOL)
    del t
    torch.cuda.empty_cache()
