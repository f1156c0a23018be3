"""The benchmark's accounting on the CPU: algorithmic bytes against a
brute-force count, the reduced ncu workloads' scale factors, and the link
between the committed ncu summaries and the kernel sources they were taken
on."""
import os

import numpy as np
import pytest

import bench
import inputs


def brute_force_bytes(w, o_bytes):
    """Every kept (query, kv head, rank) entry, and every distinct kept
    (kv head, sequence, block) with its live keys, counted one by one."""
    elt = 2 if w.kv_dtype == "bf16" else 4
    units = set()
    edges = 0
    for b in range(w.batch):
        lk = max(int(w.used_kv_lens[b]), 0) if w.pass_used else w.msb * w.block_size
        for i in range(int(w.cu_seqlens_q[b]), int(w.cu_seqlens_q[b + 1])):
            for h in range(w.hkv):
                for r in range(w.topk):
                    blk = int(w.selected[i, h, r])
                    if blk < 0 or blk * w.block_size >= lk:
                        continue
                    edges += 1
                    units.add((h, b, blk))
    keys = 0
    for h, b, blk in units:
        lk = max(int(w.used_kv_lens[b]), 0) if w.pass_used else w.msb * w.block_size
        for p in range(blk * w.block_size, min((blk + 1) * w.block_size, lk)):
            keys += int(w.block_tables[b, p // w.page_size] >= 0)
    kv = 2 * keys * w.head_dim * elt
    parts = edges * w.qhead * (w.head_dim * o_bytes + 8)
    return kv, parts, edges


@pytest.mark.parametrize("name", ["tiny", "gqa_decode", "skewed", "chunked_prefill_bf16"])
@pytest.mark.parametrize("o_bytes", [4, 2])
def test_algorithmic_bytes_brute_force(name, o_bytes):
    w = inputs.small(name, seed=3)
    got = bench.algorithmic_bytes(w, o_bytes=o_bytes)
    kv, parts, edges = brute_force_bytes(w, o_bytes)
    assert got["kv"] == kv and got["partials_write"] == parts and got["edges"] == edges
    q = out = w.tq * w.hq * w.head_dim * 4
    assert got["forward"] == kv + q + parts
    assert got["step"] == kv + q + 2 * parts + out
    fused = bench.algorithmic_bytes(w, fused=True)
    assert fused["partials_write"] == 0 and fused["forward"] == kv + q + out + fused["inv"]


@pytest.mark.parametrize("full,reduced,ratio,tol", [
    ("chunked_prefill", "chunked_prefill_ncu", 4.0, 1e-9),
    ("chunked_prefill_bf16", "chunked_prefill_bf16_ncu", 4.0, 1e-9),
    ("skewed", "skewed_ncu", 4.0, 0.01)])
def test_reduced_capture_workloads_scale(full, reduced, ratio, tol):
    """The ncu captures run on a quarter of the sequences; their traffic is
    scaled to a full launch by the ratio of algorithmic bytes, which must be
    what the profiles state."""
    a = bench.algorithmic_bytes(bench.make_workload(full, 0))["forward"]
    b = bench.algorithmic_bytes(bench.make_workload(reduced, 0))["forward"]
    assert abs(a / b - ratio) <= tol * ratio


@pytest.mark.parametrize("kernel,workload", [
    ("fused_dec.cu", "gqa_decode"), ("fused_dec.cu", "long_decode"),
    ("forward_tc.cu", "chunked_prefill"), ("forward_tc.cu", "chunked_prefill_bf16"),
    ("forward_tc.cu", "skewed"), ("forward_tc.cu", "chunked_prefill_bf16p")])
def test_profiles_match_kernel_sources(kernel, workload):
    """Each benchmark workload's ncu summary was taken on the kernel source as
    committed (its recorded hash matches), so the traffic the benchmark
    reports is that of the code it runs."""
    assert os.path.exists(os.path.join(bench.ROOT, "profiles",
                                       f"{kernel.split('.')[0]}_{workload}.md"))
    t = bench.ncu_traffic(kernel, workload)
    assert t is not None and t > 0, f"profile of {kernel} on {workload} is stale: re-capture it"


def test_code_digest_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) {  /* note */\n  return x + 1;  // one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// another header\n\nint f(int x) {\n  return x + 1;\n}\n/* tail\n   note */\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_digest(str(a)) == bench.code_digest(str(b))
    assert bench.code_digest(str(a)) != bench.code_digest(str(c))


@pytest.mark.parametrize("name", ["gqa_decode", "chunked_prefill", "skewed",
                                  "chunked_prefill_bf16", "long_decode"])
def test_cpu_baseline_shards_are_independent_sub_problems(orc, name):
    """The CPU baseline's shards (sequence, kv head, query rows) reproduce the
    whole problem's outputs for their rows: the oracle on a shard equals the
    oracle on the full workload, so the baseline times real work of the
    workload (and a sub-range of a causal sequence keeps each query's
    limit)."""
    w = inputs.small(name, seed=2)
    full_out, full_lse, _, _ = orc.attention(w.q_host(), w.k_host(), w.v_host(), w.selected,
                                             w.block_tables, w.cu_seqlens_q, w.used, w.hq,
                                             w.head_dim, w.block_size, w.page_size,
                                             w.softmax_scale, w.causal)
    row_block = 16 if w.tq > 2 * w.batch else 1
    shards = bench.shard_costs(w, row_block)
    assert sum(s[3] for s in shards) == w.tq * w.hkv
    cu = w.cu_seqlens_q
    for b, h, a, n, _ in shards[:: max(1, len(shards) // 12)]:
        s = bench.make_shard(w, b, h, a, n)
        out, lse, _, _ = orc.attention(s["q"], s["k"], s["v"], s["sel"], s["bt"], s["cu"],
                                       s["used"], s["hq"], w.head_dim, w.block_size, w.page_size,
                                       w.softmax_scale, w.causal)
        rows = np.arange(int(cu[b]) + a, int(cu[b]) + a + n)
        ref = full_out[rows][:, h * w.qhead:(h + 1) * w.qhead]
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), (b, h, a, n)
        ref_lse = full_lse[rows][:, h * w.qhead:(h + 1) * w.qhead]
        assert np.array_equal(np.isfinite(lse), np.isfinite(ref_lse))
        fin = np.isfinite(ref_lse)
        assert np.allclose(lse[fin], ref_lse[fin], rtol=1e-12, atol=1e-12)


def test_cpu_baseline_runs_threads(orc):
    w = inputs.small("skewed", seed=1)
    args = type("A", (), {"cpu_seconds": 0.2})()
    r = bench.cpu_baseline(w, args)
    assert r["kind"] == "oracle" and r["value"] > 0 and r["cores"] >= 1
    assert set(r["rates"]) == {"index", "partials_combine", "direct"}
