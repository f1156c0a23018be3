"""The fused decode path (forward and combine as one kernel, partials kept on
chip) against the oracle: batches of one query per sequence, f32 and bf16
K/V, page and block shapes the kernel supports, empty sequences, page holes,
padding, a block selected at two ranks, one or many pieces per (query, kv
head), and repeated calls on one index."""
import numpy as np
import pytest
import torch

import _gpu
import block_sparse_paged_csr_gb300 as sa
import inputs
import oracle

pytestmark = pytest.mark.gpu


def decode_case(dt, bs, ps, qhead, seed, topk=6, batch=7, pass_used=True):
    kv_min = max(900, bs * (topk + 1))                     # room for topk distinct blocks
    w = inputs.gqa_decode(seed=seed, batch=batch, kv_min=kv_min, kv_max=kv_min + 1200, hkv=2,
                          hq=2 * qhead, head_dim=128, page_size=ps, block_size=bs, topk=topk,
                          kv_dtype=dt)
    ppb = bs // ps
    blk = int(w.selected[1, 0, 0])
    w.block_tables[1, blk * ppb + ppb // 2] = -1           # a hole inside a selected block
    w.selected[3, 1, 2] = w.selected[3, 1, 1]              # one block at two ranks
    w.selected[4, 0, :] = -1                               # a (query, kv head) with no rank
    w.selected[5, 1, 1] = -1
    qo = w.qo_lens.copy()
    qo[2] = 0                                              # an empty sequence
    w.selected = np.delete(w.selected, 2, axis=0)
    w.qo_lens = qo
    w.pass_used = pass_used
    return w


def oracle_out(w, split):
    out, lse, idx, _ = oracle.attention(w.q_host(), w.k_host(), w.v_host(), w.selected,
                                        w.block_tables, w.cu_seqlens_q, w.used, w.hq,
                                        w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                                        w.causal, split_edges=split)
    return out, lse, idx


SHAPES = [("f32", 64, 16, 4), ("f32", 32, 8, 2), ("f32", 128, 16, 1), ("f32", 128, 128, 4),
          ("f32", 16, 16, 3), ("bf16", 64, 16, 8), ("bf16", 32, 16, 4), ("bf16", 128, 32, 16),
          ("bf16", 64, 8, 1), ("bf16", 256, 32, 5)]


@pytest.mark.parametrize("split", [0, 1, 6])
@pytest.mark.parametrize("dt,bs,ps,qhead", SHAPES)
def test_fused_decode_shapes(dt, bs, ps, qhead, split):
    w = decode_case(dt, bs, ps, qhead, seed=bs + ps + qhead)
    assert _gpu.uses_fused(w)
    t = _gpu.device_workload(w)
    out, lse, idx, _ = _gpu.run_attention(w, t, split_edges=split)
    ref_out, ref_lse, ref_idx = oracle_out(w, split)
    _gpu.compare_index(idx.to_host(), ref_idx)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= _gpu.TOL_F32
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, _gpu.TOL_F32)
    # the (query, kv head) without ranks (query 3 after the empty sequence):
    # zero rows, lse -inf
    qh = w.qhead
    assert torch.all(out[3, :qh] == 0) and torch.all(torch.isneginf(lse[3, :qh]))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_fused_decode_many_ranks_and_no_used(dt):
    """topk above 64 (several pieces even at the largest piece size) and
    used_kv_lens = None (every block of the table row is addressable)."""
    w = decode_case(dt, 64, 16, 4, seed=91, topk=20, pass_used=False)
    w.selected = np.concatenate([w.selected] * 4, axis=2)        # topk 80, blocks repeated
    w.topk = 80
    t = _gpu.device_workload(w)
    for split in (0, 64, 7):
        out, lse, idx, _ = _gpu.run_attention(w, t, split_edges=split)
        ref_out, ref_lse, ref_idx = oracle_out(w, split)
        _gpu.compare_index(idx.to_host(), ref_idx)
        assert _gpu.row_error(out.cpu().numpy(), ref_out) <= _gpu.TOL_F32
        _gpu.compare_lse(lse.cpu().numpy(), ref_lse, _gpu.TOL_F32)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_fused_decode_more_pairs_than_sms(dt):
    """Enough (query, kv head) pairs for whole-pair pieces on every SM plus a
    last, partial round whose pairs are cut into pieces."""
    w = decode_case(dt, 64, 16, 4, seed=23, batch=101)
    assert w.tq * w.hkv > 152
    t = _gpu.device_workload(w)
    out, lse, idx, _ = _gpu.run_attention(w, t)
    ref_out, ref_lse, ref_idx = oracle_out(w, 0)
    _gpu.compare_index(idx.to_host(), ref_idx)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= _gpu.TOL_F32
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, _gpu.TOL_F32)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_fused_decode_repeated_calls_on_one_index(dt):
    """sa_forward_combine twice on one index (the per-pair piece counters
    must be back at zero) and through sa_attention: identical results."""
    w = decode_case(dt, 64, 16, 4 if dt == "f32" else 8, seed=5)
    t = _gpu.device_workload(w)
    out0, lse0, idx, parts = _gpu.run_attention(w, t, split_edges=2)
    for _ in range(2):
        out, lse, _ = sa.sa_forward_combine(t["q"], t["k"], t["v"], idx, t["selected"],
                                            w.cu_seqlens_q, t["cu"], t["used"], t["bt"], w.hq,
                                            w.head_dim, w.block_size, w.page_size,
                                            w.softmax_scale, w.causal, split_edges=2,
                                            partials=parts)
        assert sa.sa_get_status(idx) == 0
        assert torch.equal(out, out0) and torch.equal(lse, lse0)


def test_fused_decode_matches_unfused_path():
    """The fused kernel and forward + combine (PATH_TENSOR_CORE picks the
    bf16 warp-MMA forward, PATH_CUDA_CORE the f32 one) agree to rounding."""
    for dt, qhead, path in (("f32", 4, sa.PATH_CUDA_CORE), ("bf16", 8, sa.PATH_TENSOR_CORE)):
        w = decode_case(dt, 64, 16, qhead, seed=17)
        t = _gpu.device_workload(w)
        out_f, lse_f, _, _ = _gpu.run_attention(w, t, path=sa.PATH_FUSED_DECODE)
        out_u, lse_u, _, _ = _gpu.run_attention(w, t, path=path)
        assert _gpu.row_error(out_f.cpu().numpy(), out_u.cpu().numpy()) <= _gpu.TOL_F32
        fin = torch.isfinite(lse_u)
        assert torch.equal(fin, torch.isfinite(lse_f))
        assert torch.max(torch.abs(lse_f[fin] - lse_u[fin])).item() <= 1e-4


def test_fused_decode_path_refusals():
    w = inputs.small("chunked_prefill", seed=0)      # several queries per sequence
    t = _gpu.device_workload(w)
    with pytest.raises(sa.SAError) as e:
        _gpu.run_attention(w, t, path=sa.PATH_FUSED_DECODE)
    assert e.value.kind == "UNSUPPORTED"
    d = decode_case("f32", 64, 16, 4, seed=3)
    td = _gpu.device_workload(d)
    idx = sa.sa_build_index(td["selected"], d.cu_seqlens_q, td["cu"], td["used"], d.max_pages,
                            d.block_size, d.page_size)
    with pytest.raises(sa.SAError) as e:
        sa.sa_forward(td["q"], td["k"], td["v"], idx, td["bt"], td["cu"], td["used"], d.hq, d.hkv,
                      d.head_dim, d.block_size, d.page_size, d.softmax_scale, d.causal,
                      path=sa.PATH_FUSED_DECODE)
    assert e.value.kind == "UNSUPPORTED"


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_attention_graph_replay(dt):
    """sa_attention captured into a CUDA graph (index, fused forward +
    combine) and replayed after the inputs' contents change: the same out and
    lse as eager calls on the new contents."""
    w = decode_case(dt, 64, 16, 4 if dt == "f32" else 8, seed=44)
    t = _gpu.device_workload(w)
    g = sa.AttentionGraph(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q, t["cu"],
                          t["used"], t["bt"], w.hq, w.hkv, w.head_dim, w.block_size,
                          w.page_size, w.softmax_scale, w.causal)
    rng = np.random.default_rng(3)
    for it in range(3):
        t["q"].copy_(torch.from_numpy(rng.standard_normal(tuple(t["q"].shape)).astype(np.float32)))
        sel = w.selected.copy()
        rng.shuffle(sel, axis=2)                       # the same blocks at other ranks
        t["selected"].copy_(torch.from_numpy(sel))
        out, lse = g.replay()
        torch.cuda.synchronize()
        assert sa.sa_get_status(g.index) == 0
        ref_out, ref_lse, _, _ = _gpu.run_attention(w, t)
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
