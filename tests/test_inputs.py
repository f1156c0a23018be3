"""The seeded input generators (CPU): value distribution, bf16 rounding and the
structure of the five workloads."""
import numpy as np
import pytest
import torch

import inputs


def test_counter_values_are_deterministic_and_sliceable():
    a = inputs.counter_normal(3, inputs.STREAM_K, 0, 10_000)
    b = inputs.counter_normal(3, inputs.STREAM_K, 4000, 100)
    assert np.array_equal(a[4000:4100], b)
    c = inputs.counter_normal(4, inputs.STREAM_K, 0, 10_000)
    assert not np.array_equal(a, c)


def test_counter_values_distribution():
    x = inputs.counter_normal(0, inputs.STREAM_Q, 0, 2_000_000).astype(np.float64)
    assert abs(x.mean()) < 3e-3
    assert abs(x.var() - 1.0) < 5e-3
    assert np.abs(x).max() < 3.47
    # Irwin-Hall(4) kurtosis: 3 - 6/(5*4) = 2.7
    k = np.mean(x ** 4) / np.mean(x ** 2) ** 2
    assert abs(k - 2.7) < 0.02


def test_bf16_bits_round_to_nearest_even_like_torch():
    x = inputs.counter_normal(1, inputs.STREAM_V, 0, 100_000)
    ours = inputs.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = inputs.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("name", ["tiny", "gqa_decode", "chunked_prefill", "skewed",
                                  "long_decode"])
def test_small_workload_structure(name):
    w = inputs.small(name, seed=0)
    tq, hkv, topk = w.selected.shape
    assert tq == w.tq and hkv == w.hkv and topk == w.topk
    assert w.selected.min() >= -1 and w.selected.max() < w.msb
    cu = w.cu_seqlens_q
    for i in range(tq):
        b = int(np.searchsorted(cu, i, side="right") - 1)
        for h in range(hkv):
            row = w.selected[i, h]
            live = row[row >= 0]
            assert live.size == np.unique(live).size, "blocks are distinct per (query, head)"
            lk = int(w.used_kv_lens[b])
            assert np.all(live * w.block_size < lk) or name == "skewed"
            if name == "gqa_decode":
                assert row[0] == -(-lk // w.block_size) - 1
            if name == "chunked_prefill":
                t = i - cu[b]
                assert row[0] == (lk - w.qo_lens[b] + t) // w.block_size
                assert np.all(row[1:] < row[0])
    bt = w.block_tables
    live = bt[bt >= 0]
    assert live.size == np.unique(live).size and live.max() < w.num_pages


def test_full_workload_shapes():
    d = inputs.gqa_decode(0)
    assert (d.batch, d.hq, d.hkv, d.head_dim, d.page_size, d.block_size, d.topk) == \
        (64, 32, 8, 128, 16, 64, 16)
    assert d.max_pages == 2048 and d.msb == 512 and d.num_pages == 131072
    assert d.used_kv_lens.min() >= 4096 and d.used_kv_lens.max() <= 32768
    p = inputs.chunked_prefill(0)
    assert p.tq == 8192 and p.msb == 256 and p.selected.shape == (8192, 8, 32)
    s = inputs.skewed(0)
    assert s.tq == 8192 and s.msb == 1024 and s.selected.shape == (8192, 4, 24)
    pad = np.mean(s.selected < 0)
    assert 0.13 < pad < 0.17
    # a few blocks receive hundreds of edges per (head, sequence)
    h0 = s.selected[:512, 0].ravel()
    counts = np.bincount(h0[h0 >= 0])
    assert counts.max() > 300
    l = inputs.long_decode(0)
    assert l.num_pages == 128 * 8192 and l.kv_dtype == "bf16" and l.msb == 2048
    assert 0.08 < np.mean(l.selected < 0) < 0.12
