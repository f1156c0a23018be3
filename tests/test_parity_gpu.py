"""Parity of the CUDA library (through its C ABI) with the oracle.

* Index: bit-exact, every array, on every workload shape and random edge cases.
* Partials and outputs: element by element within the f32 tolerance (1e-4,
  row-normalised) on reduced workloads the oracle finishes in seconds.
* Full-size serving workloads (the launch configuration the benchmark times):
  the index bit-exact, outputs on sampled (query, q-head) rows recomputed by
  the oracle's query-outer attention.
"""
import numpy as np
import pytest
import torch

import _gpu
import _pins
import block_sparse_paged_csr_gb300 as sa
import inputs
import oracle

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "gqa_decode", "chunked_prefill", "chunked_prefill_bf16", "skewed",
         "long_decode"]


def _oracle_attention(w, split_edges):
    return oracle.attention(w.q_host(), w.k_host(), w.v_host(), w.selected, w.block_tables,
                            w.cu_seqlens_q, w.used, w.hq, w.head_dim, w.block_size, w.page_size,
                            w.softmax_scale, w.causal, split_edges=split_edges)


@pytest.mark.parametrize("split", [0, 3])
@pytest.mark.parametrize("name", SMALL)
def test_small_workload_parity(name, split):
    w = inputs.small(name, seed=0)
    t = _gpu.device_workload(w)
    out, lse, idx, (o, m, l) = _gpu.run_attention(w, t, split_edges=split)
    ref_out, ref_lse, ref_idx, (ro, rm, rl) = _oracle_attention(w, split)
    _gpu.compare_index(idx.to_host(), ref_idx)
    rows = ref_idx["edges"].shape[0] * w.qhead
    tol = _gpu.auto_tol(w)
    if not _gpu.uses_fused(w):      # the fused decode path keeps its partials on chip
        _gpu.compare_partials(o[:rows].cpu().numpy(), m[:rows].cpu().numpy(),
                              l[:rows].cpu().numpy(), ro, rm, rl, tol)
        _gpu.report(f"small {name} split {split}", "o_partial", o[:rows].cpu().numpy(), ro)
        _gpu.report(f"small {name} split {split}", "l_partial", l[:rows].cpu().numpy(), rl)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= tol
    _gpu.report(f"small {name} split {split}", "out", out.cpu().numpy(), ref_out)
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, tol)


def _case_tensors(c, dev="cuda"):
    k, v = c["k"], c["v"]
    if k.dtype == np.uint16:
        kt = torch.from_numpy(k.view(np.int16)).to(dev).view(torch.bfloat16)
        vt = torch.from_numpy(v.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        kt, vt = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    return dict(q=torch.from_numpy(c["q"]).to(dev), k=kt, v=vt,
                selected=torch.from_numpy(c["sel"]).to(dev),
                cu=torch.from_numpy(c["cu"]).to(dev),
                used=None if c["used"] is None else torch.from_numpy(c["used"]).to(dev),
                bt=torch.from_numpy(c["bt"]).to(dev))


@pytest.mark.parametrize("seed", range(24))
def test_random_edge_cases(seed):
    """Empty sequences, page holes (-1), blocks past the KV length, repeated
    blocks, used_kv_lens = None, GQA, several pages per block, both masks."""
    bf16 = seed % 3 == 0
    c = _pins.random_case(seed, bf16=bf16, full=bool(seed % 2))
    if bf16 and c["d"] % 8:
        c = _pins.random_case(seed + 100, bf16=True, full=bool(seed % 2))
        if c["d"] % 8:
            pytest.skip("bf16 needs head_dim % 8 == 0")
    if seed % 5 == 0 and c["sel"].shape[2] > 1:
        c["sel"][..., 1] = c["sel"][..., 0]
    t = _case_tensors(c)
    for causal in (False, True):
        split = seed % 3
        out, lse, idx, (o, m, l) = sa.sa_attention(
            t["q"], t["k"], t["v"], t["selected"], c["cu"], t["cu"], t["used"], t["bt"], c["hq"],
            c["hkv"], c["d"], c["bs"], c["ps"], c["scale"], causal, split_edges=split)
        assert sa.sa_get_status(idx) == 0
        ref_out, ref_lse, ref_idx, (ro, rm, rl) = oracle.attention(
            c["q"], c["k"], c["v"], c["sel"], c["bt"], c["cu"], c["used"], c["hq"], c["d"],
            c["bs"], c["ps"], c["scale"], causal, split_edges=split)
        _gpu.compare_index(idx.to_host(), ref_idx)
        rows = ref_idx["edges"].shape[0] * (c["hq"] // c["hkv"])
        num_pages = t["k"].numel() // (c["hkv"] * c["ps"] * c["d"])
        fused = sa.sa_attention_kernel_name(
            c["cu"], num_pages, c["hkv"], c["hq"], c["d"], c["bs"], c["ps"],
            "bf16" if bf16 else "f32") == "fused_dec_kernel"
        if not fused:
            _gpu.compare_partials(o[:rows].cpu().numpy(), m[:rows].cpu().numpy(),
                                  l[:rows].cpu().numpy(), ro, rm, rl, _gpu.TOL_F32)
        assert _gpu.row_error(out.cpu().numpy(), ref_out) <= _gpu.TOL_F32
        _gpu.compare_lse(lse.cpu().numpy(), ref_lse, _gpu.TOL_F32)


def test_separate_steps_match_fused():
    w = inputs.small("skewed", seed=2)
    t = _gpu.device_workload(w)
    out_f, lse_f, _, _ = _gpu.run_attention(w, t, split_edges=4)
    idx = sa.sa_build_index(t["selected"], w.cu_seqlens_q, t["cu"], t["used"], w.max_pages,
                            w.block_size, w.page_size, split_edges=4)
    o, m, l = sa.sa_forward(t["q"], t["k"], t["v"], idx, t["bt"], t["cu"], t["used"], w.hq, w.hkv,
                            w.head_dim, w.block_size, w.page_size, w.softmax_scale, w.causal)
    out, lse = sa.sa_combine(idx, o, m, l, w.hq, w.head_dim)
    assert sa.sa_get_status(idx) == 0
    assert torch.equal(out, out_f) and torch.equal(lse, lse_f)


def test_all_padding_gives_zero_output():
    w = inputs.small("gqa_decode", seed=3)
    w.selected[:] = -1
    t = _gpu.device_workload(w)
    out, lse, idx, _ = _gpu.run_attention(w, t)
    assert int(idx.totals[0]) == 0
    assert torch.count_nonzero(out) == 0
    assert torch.all(torch.isneginf(lse))


def test_device_detected_errors_are_reported():
    w = inputs.small("tiny", seed=0)
    t = _gpu.device_workload(w)
    bad = t["selected"].clone()
    bad[1, 0, 1] = w.msb                                   # outside [-1, msb)
    _, _, idx, _ = sa.sa_attention(t["q"], t["k"], t["v"], bad, w.cu_seqlens_q, t["cu"],
                                   t["used"], t["bt"], w.hq, w.hkv, w.head_dim, w.block_size,
                                   w.page_size, w.softmax_scale, w.causal)
    assert sa.sa_get_status(idx) == 5                      # SELECTED_RANGE
    bt = t["bt"].clone()
    blk = int(w.selected[0, 0, 0])
    bt[0, blk * w.ppb] = w.num_pages                       # page id == num_pages
    _, _, idx, _ = sa.sa_attention(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q, t["cu"],
                                   t["used"], bt, w.hq, w.hkv, w.head_dim, w.block_size,
                                   w.page_size, w.softmax_scale, w.causal)
    assert sa.sa_get_status(idx) == 4                      # SHAPE
    # a clean call afterwards reports nothing
    _, _, idx, _ = _gpu.run_attention(w, t)


def test_host_checks_raise():
    w = inputs.small("tiny", seed=0)
    t = _gpu.device_workload(w)
    with pytest.raises(sa.SAError, match="HEAD_COUNT"):
        sa.sa_attention(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q, t["cu"], t["used"],
                        t["bt"], 3, w.hkv, w.head_dim, w.block_size, w.page_size, 0.1, False)
    with pytest.raises(sa.SAError, match="SHAPE"):
        bad_cu = w.cu_seqlens_q.copy()
        bad_cu[-1] += 1
        sa.sa_build_index(t["selected"], bad_cu, t["cu"], t["used"], w.max_pages, w.block_size,
                          w.page_size)


def test_device_fill_matches_host_generator():
    for dtype in ("f32", "bf16"):
        n = 1 << 20
        dev = torch.empty(n, dtype=torch.float32 if dtype == "f32" else torch.bfloat16,
                          device="cuda")
        inputs.fill_device(dev, 7, inputs.STREAM_V, start=12345, bf16=dtype == "bf16")
        host = inputs.counter_normal(7, inputs.STREAM_V, 12345, n)
        if dtype == "bf16":
            got = dev.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, inputs.bf16_bits(host))
        else:
            assert np.array_equal(dev.cpu().numpy(), host)


# --------------------------------------------------------------------------- full size

FULL = ["gqa_decode", "chunked_prefill", "chunked_prefill_bf16", "skewed", "long_decode"]
SPLIT = {"gqa_decode": 0, "chunked_prefill": 16, "chunked_prefill_bf16": 16, "skewed": 16,
         "long_decode": 0}


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """The serving workloads at full size: index bit-exact against the oracle,
    outputs on sampled rows against the oracle's query-outer attention."""
    w = inputs.FULL[name](0)
    t = _gpu.device_workload(w, fill_on_device=True)
    out, lse, idx, parts = _gpu.run_attention(w, t, split_edges=SPLIT[name])
    ref_idx = oracle.build_index(w.selected, w.cu_seqlens_q, w.used, w.max_pages, w.block_size,
                                 w.page_size, SPLIT[name])
    _gpu.compare_index(idx.to_host(), ref_idx)
    rng = np.random.default_rng(11)
    n_q = 6 if name == "long_decode" else 12
    queries = np.unique(rng.choice(w.tq, size=n_q, replace=False))
    k, v, bt, num_pages = w.compact_pool(queries)
    rows = np.array([(i, hq) for i in queries for hq in rng.choice(w.hq, 4, replace=False)])
    q = w.q_host()
    ref, ref_lse = oracle.direct(q, k, v, w.selected, bt, w.cu_seqlens_q, w.used, w.hq,
                                 w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                                 w.causal, rows=rows)
    got = out[rows[:, 0], rows[:, 1]].cpu().numpy()
    tol = _gpu.auto_tol(w)
    assert _gpu.row_error(got, ref) <= tol
    _gpu.report(f"full {name} sampled rows", "out", got, ref)
    _gpu.compare_lse(lse[rows[:, 0], rows[:, 1]].cpu().numpy(), ref_lse, tol)
    if not _gpu.uses_fused(w):
        _check_hot_units(w, idx.to_host(), parts, 8 if name == "skewed" else 1, tol, name)
    del t
    torch.cuda.empty_cache()


def _check_hot_units(w, ih, parts, n_units, tol, name):
    """Every partial row of the n_units units with the most edges, against the
    oracle's query-outer attention over that unit's block alone (a one-block
    selection: out = o / l, lse = m + log l of the partial)."""
    o_p, m_p, l_p = parts
    q = w.q_host()
    cand = []
    for h in range(w.hkv):
        offs = ih["sel_offsets"][h]
        cnt = np.diff(offs[: int(ih["num_sel"][h]) + 1])
        for j in np.argsort(-cnt, kind="stable")[:n_units]:
            cand.append((int(cnt[j]), h, int(j)))
    cand.sort(key=lambda c: -c[0])
    for cnt, h, j in cand[:n_units]:
        raw = int(ih["sel_slots"][h, j])
        b, blk = divmod(raw, w.msb)
        e0 = int(ih["edge_head_base"][h]) + int(ih["sel_offsets"][h, j])
        edges = ih["edges"][e0:e0 + cnt]
        pages = w.block_tables[b, blk * w.ppb:(blk + 1) * w.ppb]
        live = pages >= 0
        k, v = w.k_host(pages[live]), w.v_host(pages[live])
        bt = np.full_like(w.block_tables, -1)
        bt[b, blk * w.ppb:(blk + 1) * w.ppb][live] = np.arange(int(live.sum()), dtype=np.int32)
        sel1 = np.full((w.tq, w.hkv, 1), -1, np.int32)
        sel1[edges[:, 0], h, 0] = blk
        rows = np.array([(int(i), h * w.qhead + qh) for i, _ in edges for qh in range(w.qhead)])
        ref, ref_lse = oracle.direct(q, k, v, sel1, bt, w.cu_seqlens_q, w.used, w.hq,
                                     w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                                     w.causal, rows=rows)
        prow = (np.arange(e0, e0 + cnt)[:, None] * w.qhead + np.arange(w.qhead)[None, :]).ravel()
        sel_rows = torch.from_numpy(prow).to(o_p.device)
        o = o_p[sel_rows].float().cpu().numpy().astype(np.float64)
        m = m_p[sel_rows].cpu().numpy().astype(np.float64)
        l = l_p[sel_rows].cpu().numpy().astype(np.float64)
        live_rows = l > 0
        assert np.array_equal(live_rows, np.isfinite(ref_lse)), "empty partial rows differ"
        got = np.zeros_like(o)
        got[live_rows] = o[live_rows] / l[live_rows, None]
        assert _gpu.row_error(got, ref) <= tol, f"unit ({h}, {raw}) with {cnt} edges"
        _gpu.report(f"full {name} unit of {cnt} edges", "o/l", got, ref)
        lse_got = np.where(live_rows, m + np.log(np.where(live_rows, l, 1.0)), -np.inf)
        _gpu.compare_lse(lse_got, ref_lse, tol)


# --------------------------------------------------------------------------- each kernel


def _check_against_oracle(w, t, split, path, tol=_gpu.TOL_F32, report=None):
    out, lse, idx, (o, m, l) = _gpu.run_attention(w, t, split_edges=split, path=path)
    ref_out, ref_lse, ref_idx, (ro, rm, rl) = _oracle_attention(w, split)
    _gpu.compare_index(idx.to_host(), ref_idx)
    rows = ref_idx["edges"].shape[0] * w.qhead
    _gpu.compare_partials(o[:rows].cpu().numpy(), m[:rows].cpu().numpy(), l[:rows].cpu().numpy(),
                          ro, rm, rl, tol)
    assert _gpu.row_error(out.cpu().numpy(), ref_out) <= tol
    _gpu.compare_lse(lse.cpu().numpy(), ref_lse, tol)
    if report:
        _gpu.report(report, "o_partial", o[:rows].cpu().numpy(), ro)
        _gpu.report(report, "out", out.cpu().numpy(), ref_out)


@pytest.mark.parametrize("split", [0, 2])
@pytest.mark.parametrize("path", [sa.PATH_CUDA_CORE, sa.PATH_CUDA_CORE_GENERAL],
                         ids=["cuda_core", "cuda_core_general"])
@pytest.mark.parametrize("name", SMALL)
def test_small_workload_each_cuda_core_kernel(name, path, split):
    """PATH_CUDA_CORE runs the pipelined decode kernel wherever its limits
    allow (head_dim 128), including multi-edge splits (row groups);
    PATH_CUDA_CORE_GENERAL the general kernel."""
    w = inputs.small(name, seed=1)
    _check_against_oracle(w, _gpu.device_workload(w), split, path)


@pytest.mark.parametrize("bs,ps,qhead,dt", [(32, 16, 1, "f32"), (64, 16, 2, "bf16"),
                                            (128, 64, 8, "f32"), (128, 16, 8, "bf16"),
                                            (64, 8, 4, "f32"), (32, 4, 4, "bf16"),
                                            (64, 16, 8, "f32"), (128, 32, 4, "bf16")])
def test_decode_kernel_shapes(bs, ps, qhead, dt):
    w = inputs.gqa_decode(seed=bs + ps + qhead, batch=7, kv_min=900, kv_max=2100, hkv=2,
                          hq=2 * qhead, head_dim=128, page_size=ps, block_size=bs, topk=6,
                          kv_dtype=dt)
    w.block_tables[1, 3] = -1          # a hole inside a live block
    _check_against_oracle(w, _gpu.device_workload(w), 0, sa.PATH_CUDA_CORE)


# --------------------------------------------------------------------------- tensor cores

TC_SMALL = ["gqa_decode", "chunked_prefill", "chunked_prefill_bf16", "skewed", "long_decode"]


TC_PATHS = {"bf16_operands": sa.PATH_TENSOR_CORE, "tf32_scores": sa.PATH_TENSOR_CORE_TF32}


@pytest.mark.parametrize("path", list(TC_PATHS), ids=list(TC_PATHS))
@pytest.mark.parametrize("split", [0, 3, 16])
@pytest.mark.parametrize("name", TC_SMALL)
def test_small_workload_tensor_core(name, split, path):
    """The tcgen05 kernel on every reduced workload it supports, with every
    operand rounded to bf16 (SA_PATH_TENSOR_CORE) and with the scores from
    Q and K kept f32 (tf32 operands) for f32 K/V (SA_PATH_TENSOR_CORE_TF32);
    split 0 puts whole units (more than 128 rows) in one split, so row tiles
    repeat.  The measured errors of both are in the session's report."""
    w = inputs.small(name, seed=2)
    _check_against_oracle(w, _gpu.device_workload(w), split, TC_PATHS[path], _gpu.TOL_TC,
                          report=f"small {name} {path} split {split}")


@pytest.mark.parametrize("path", list(TC_PATHS), ids=list(TC_PATHS))
@pytest.mark.parametrize("bs,ps,qhead,dt,causal", [(64, 16, 8, "f32", True),
                                                   (128, 64, 8, "bf16", True),
                                                   (64, 8, 4, "bf16", False),
                                                   (128, 32, 2, "f32", True),
                                                   (64, 64, 1, "f32", False),
                                                   (128, 16, 16, "bf16", True),
                                                   (128, 128, 8, "f32", False)])
def test_tensor_core_shapes(bs, ps, qhead, dt, causal, path):
    w = inputs.chunked_prefill(seed=bs + ps + qhead, batch=3, qo_len=30, kv_len=1500, hkv=2,
                               hq=2 * qhead, head_dim=128, page_size=ps, block_size=bs, topk=5,
                               kv_dtype=dt)
    w.causal = causal
    w.block_tables[1, 2] = -1              # a hole inside a live block
    _check_against_oracle(w, _gpu.device_workload(w), 7, TC_PATHS[path], _gpu.TOL_TC)


@pytest.mark.parametrize("bs,ps,qhead", [(64, 16, 8), (32, 16, 1), (128, 64, 4), (64, 8, 2),
                                         (128, 16, 16), (64, 32, 8)])
def test_decode_mma_shapes(bs, ps, qhead):
    """bf16 decode on warp-level MMA (split bf16 operands): f32-class
    accuracy, including repeated blocks (multi-edge units -> row groups)."""
    w = inputs.gqa_decode(seed=3 * bs + ps + qhead, batch=7, kv_min=900, kv_max=2100, hkv=2,
                          hq=2 * qhead, head_dim=128, page_size=ps, block_size=bs, topk=6,
                          kv_dtype="bf16")
    w.block_tables[2, 1] = -1
    w.selected[3, 1, 2] = w.selected[3, 1, 1]      # a block selected at two ranks
    _check_against_oracle(w, _gpu.device_workload(w), 0, sa.PATH_TENSOR_CORE, _gpu.TOL_F32)


@pytest.mark.parametrize("name", ["chunked_prefill", "chunked_prefill_bf16", "skewed"])
def test_tensor_core_bf16_q_copy_matches_f32_gather(name):
    """sa_attention lets the tensor-core forward gather Q from a bf16 copy it
    keeps in `out` until the combine; sa_forward gathers the f32 rows and
    rounds them itself.  Same rounding, so the partials are bit-identical;
    and an `out` that is q itself (no room for the copy) gives the same
    output."""
    w = inputs.small(name, seed=9)
    t = _gpu.device_workload(w)
    path = sa.PATH_TENSOR_CORE                 # bf16 operands: the path that uses the copy
    out, lse, idx, (o, m, l) = _gpu.run_attention(w, t, split_edges=3, path=path)
    o2, m2, l2 = sa.sa_forward(t["q"], t["k"], t["v"], idx, t["bt"], t["cu"], t["used"], w.hq,
                               w.hkv, w.head_dim, w.block_size, w.page_size, w.softmax_scale,
                               w.causal, path=path)
    assert sa.sa_get_status(idx) == 0
    rows = int(idx.to_host()["edges"].shape[0]) * w.qhead
    assert torch.equal(o[:rows], o2[:rows])
    assert torch.equal(m[:rows], m2[:rows]) and torch.equal(l[:rows], l2[:rows])
    q_alias = t["q"].clone()
    out3, lse3, _, _ = sa.sa_attention(q_alias, t["k"], t["v"], t["selected"], w.cu_seqlens_q,
                                       t["cu"], t["used"], t["bt"], w.hq, w.hkv, w.head_dim,
                                       w.block_size, w.page_size, w.softmax_scale, w.causal,
                                       split_edges=3, out=q_alias, path=path)
    torch.cuda.synchronize()
    assert torch.equal(out3, out) and torch.equal(lse3, lse)


LEFT_PATHS = {"auto": sa.PATH_AUTO, "cuda_core": sa.PATH_CUDA_CORE,
              "cuda_core_general": sa.PATH_CUDA_CORE_GENERAL,
              "tensor_core": sa.PATH_TENSOR_CORE}


@pytest.mark.parametrize("path", list(LEFT_PATHS), ids=list(LEFT_PATHS))
@pytest.mark.parametrize("name", ["gqa_decode", "chunked_prefill", "chunked_prefill_bf16",
                                  "skewed", "long_decode"])
def test_left_aligned_causal(name, path):
    """causal = 2 (left-aligned: key p live for the t-th query of its chunk
    iff p <= t) on every kernel; decode batches leave the fused path (a lone
    query then sees key 0 at most)."""
    w = inputs.small(name, seed=12)
    w.causal = 2
    p = LEFT_PATHS[path]
    kernel = sa.sa_attention_kernel_name(w.cu_seqlens_q, w.num_pages, w.hkv, w.hq, w.head_dim,
                                         w.block_size, w.page_size, w.kv_dtype, path=p, causal=2)
    if kernel is None:
        pytest.skip("no kernel of this path for the shape")
    assert kernel != "fused_dec_kernel"
    tol = _gpu.TOL_TC if kernel == "forward_tc_kernel" or path == "tensor_core" else _gpu.TOL_F32
    _check_against_oracle(w, _gpu.device_workload(w), 3, p, tol)


@pytest.mark.parametrize("name", ["chunked_prefill", "skewed"])
def test_attention_graph_replay_unfused(name):
    """The unfused path (index, Q rounding pass, tensor-core forward,
    combine) captured into a CUDA graph: replays after the queries change
    equal eager calls."""
    w = inputs.small(name, seed=13)
    t = _gpu.device_workload(w)
    g = sa.AttentionGraph(t["q"], t["k"], t["v"], t["selected"], w.cu_seqlens_q, t["cu"],
                          t["used"], t["bt"], w.hq, w.hkv, w.head_dim, w.block_size,
                          w.page_size, w.softmax_scale, w.causal, split_edges=3)
    rng = np.random.default_rng(4)
    for _ in range(2):
        t["q"].copy_(torch.from_numpy(rng.standard_normal(tuple(t["q"].shape)).astype(np.float32)))
        out, lse = g.replay()
        torch.cuda.synchronize()
        assert sa.sa_get_status(g.index) == 0
        ref_out, ref_lse, _, _ = _gpu.run_attention(w, t, split_edges=3)
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("topk,split", [(64, 0), (64, 3), (65, 3), (33, 1)])
def test_decode_index_segment_modes(topk, split):
    """The index kernel builds segments of at most 64 entries (one query per
    sequence, topk <= 64: decode batches) one warp each, larger ones through
    shared-memory histograms; both give the oracle's index bit for bit,
    with repeated blocks, -1 padding, blocks past the KV length and an empty
    sequence in the batch."""
    w = inputs.gqa_decode(seed=topk + split, batch=9, kv_min=4400, kv_max=6000, hq=8, hkv=2,
                          head_dim=32, topk=topk)
    rng = np.random.default_rng(topk)
    sel = w.selected
    sel[rng.random(sel.shape) < 0.1] = -1
    sel[2, 0, 5] = sel[2, 0, 7]                      # a block chosen at two ranks
    sel[4, 1, 3] = w.msb - 1                         # past the sequence's KV length
    w.qo_lens = w.qo_lens.copy()
    w.qo_lens[6] = 0                                 # an empty sequence
    w.selected = np.delete(sel, 6, axis=0)
    t = {"selected": torch.from_numpy(w.selected).cuda(),
         "cu": torch.from_numpy(w.cu_seqlens_q).cuda(),
         "used": torch.from_numpy(w.used_kv_lens).cuda()}
    idx = sa.sa_build_index(t["selected"], w.cu_seqlens_q, t["cu"], t["used"], w.max_pages,
                            w.block_size, w.page_size, split_edges=split)
    assert sa.sa_get_status(idx) == 0
    ref = oracle.build_index(w.selected, w.cu_seqlens_q, w.used_kv_lens, w.max_pages,
                             w.block_size, w.page_size, split)
    _gpu.compare_index(idx.to_host(), ref)
