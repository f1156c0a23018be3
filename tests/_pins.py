"""Pins of the oracle against things other than itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.lib()`` or a
deliberately altered build) and raises AssertionError (or OracleError) when the
oracle disagrees with:

* the values printed in the pages' own tests (tests/golden/types_fixtures.json);
* dense softmax attention written with numpy (query-outer, no blocks, no
  index), which must equal the sparse result whenever every block is selected
  (the "sparse full matches dense reference" fixture named in gpu.rs);
* invariances the method guarantees: permuting ranks or padding with -1
  leaves the output unchanged;
* special cases with textbook or closed-form answers: one selected block is
  plain softmax attention over that block; equal keys give the mean of the
  selected values; a one-key block gives (o = v, l = 1);
* a brute-force index built by sorting (a different construction from the
  oracle's bucket append).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- dense reference


def dense_reference(q, k, v, block_tables, cu, used, hkv, head_dim, block_size, page_size,
                    scale, causal):
    """Softmax attention of every query over all keys of its sequence.

    Keys of sequence b are the positions p < lk_b whose page
    block_tables[b, p // page_size] is not -1; with `causal`, also p <= limit
    (right-aligned; causal = 2: left-aligned, limit = the query's position in
    its chunk).  Written with numpy matrix products, query-outer."""
    q = np.asarray(q, np.float64)
    kf = oracle_free_f64(k)
    vf = oracle_free_f64(v)
    tq, hq, d = q.shape
    qhead = hq // hkv
    max_pages = block_tables.shape[1]
    msb = max_pages // (block_size // page_size)
    out = np.zeros((tq, hq, d))
    lse = np.full((tq, hq), -np.inf)
    for b in range(len(cu) - 1):
        lk = msb * block_size if used is None else max(int(used[b]), 0)
        pos = [p for p in range(min(lk, msb * block_size))
               if block_tables[b, p // page_size] >= 0]
        pages = np.array([block_tables[b, p // page_size] for p in pos], dtype=np.int64)
        rows = np.array([p % page_size for p in pos], dtype=np.int64)
        pos = np.array(pos, dtype=np.int64)
        qo = int(cu[b + 1] - cu[b])
        for t in range(qo):
            i = int(cu[b]) + t
            limit = t if causal == 2 else ((lk - qo + t) if lk >= qo else t)
            alive = np.ones(pos.size, bool) if not causal else pos <= limit
            for h in range(hkv):
                K = kf[pages, h, rows, :][alive]
                V = vf[pages, h, rows, :][alive]
                if K.shape[0] == 0:
                    continue
                Q = q[i, h * qhead:(h + 1) * qhead, :]
                S = scale * (Q @ K.T)
                M = S.max(axis=1, keepdims=True)
                P = np.exp(S - M)
                L = P.sum(axis=1, keepdims=True)
                out[i, h * qhead:(h + 1) * qhead] = (P @ V) / L
                lse[i, h * qhead:(h + 1) * qhead] = (M + np.log(L))[:, 0]
    return out, lse


def oracle_free_f64(pages):
    """Pool values as float64 (bf16 bit patterns widened exactly)."""
    a = np.asarray(pages)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def full_selection(tq, hkv, msb, rng=None, pad=0):
    """Every block once per (query, kv head), optionally shuffled and padded."""
    sel = np.tile(np.arange(msb, dtype=np.int32), (tq, hkv, 1))
    if rng is not None:
        for i in range(tq):
            for h in range(hkv):
                sel[i, h] = rng.permutation(sel[i, h])
    if pad:
        sel = np.concatenate([sel, np.full((tq, hkv, pad), -1, np.int32)], axis=2)
        if rng is not None:
            for i in range(tq):
                for h in range(hkv):
                    sel[i, h] = rng.permutation(sel[i, h])
    return sel


def fixture_f1():
    """gpu.rs, test gpu_forward_matches_cpu_forward_small."""
    tq, hq, hkv, d, ps, bs, max_pages, num_pages = 2, 1, 1, 4, 2, 2, 3, 3
    q = (np.arange(tq * hq * d, dtype=np.float32) * np.float32(0.11)).reshape(tq, hq, d)
    n = num_pages * hkv * ps * d
    k = np.sin(np.arange(n, dtype=np.float32) * np.float32(0.07)).reshape(num_pages, hkv, ps, d)
    v = np.cos(np.arange(n, dtype=np.float32) * np.float32(0.13)).reshape(num_pages, hkv, ps, d)
    bt = np.array([[0, 1, 2]], np.int32)
    cu = np.array([0, tq], np.int64)
    used = np.array([6], np.int32)
    sel = np.tile(np.arange(max_pages, dtype=np.int32), (tq, hkv, 1))
    return dict(q=q, k=k, v=v, bt=bt, cu=cu, used=used, sel=sel, hq=hq, hkv=hkv, d=d, bs=bs,
                ps=ps, scale=float(np.float32(1.0) / np.sqrt(np.float32(d))))


def fixture_f2():
    """gpu.rs, test gpu_forward_gqa_multi_batch."""
    tq, hq, hkv, d, ps, bs, max_pages, num_pages = 3, 4, 2, 8, 4, 4, 3, 3
    q = np.sin(np.arange(tq * hq * d, dtype=np.float32) * np.float32(0.05)).reshape(tq, hq, d)
    n = num_pages * hkv * ps * d
    k = np.cos(np.arange(n, dtype=np.float32) * np.float32(0.03)).reshape(num_pages, hkv, ps, d)
    v = np.sin(np.arange(n, dtype=np.float32) * np.float32(0.09)).reshape(num_pages, hkv, ps, d)
    bt = np.array([[0, 1, 2], [0, 1, 2]], np.int32)
    cu = np.array([0, 2, 3], np.int64)
    used = np.array([12, 12], np.int32)
    sel = np.tile(np.arange(max_pages, dtype=np.int32), (tq, hkv, 1))
    return dict(q=q, k=k, v=v, bt=bt, cu=cu, used=used, sel=sel, hq=hq, hkv=hkv, d=d, bs=bs,
                ps=ps, scale=float(np.float32(1.0) / np.sqrt(np.float32(d))))


def random_case(seed, bf16=False, holes=True, pass_used=True, full=True, allow_empty_seq=True):
    """A tiny random problem: several sequences (some may be empty), GQA,
    several pages per block, page holes (-1), ragged KV lengths."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    qo = rng.integers(0 if allow_empty_seq else 1, 5, size=B)
    if qo.sum() == 0:
        qo[0] = 1
    hkv = int(rng.integers(1, 4))
    qhead = int(rng.integers(1, 4))
    hq = hkv * qhead
    d = int(rng.choice([4, 8]))
    ps = int(rng.choice([1, 2, 3]))
    ppb = int(rng.integers(1, 4))
    bs = ps * ppb
    msb = int(rng.integers(2, 6))
    max_pages = msb * ppb + int(rng.integers(0, ppb))  # may leave a partial block unaddressable
    num_pages = B * max_pages + 2
    perm = rng.permutation(num_pages)[: B * max_pages].astype(np.int32).reshape(B, max_pages)
    if holes:
        perm[rng.random(perm.shape) < 0.15] = -1
    lens = rng.integers(0, msb * bs + 1, size=B).astype(np.int32)
    lens[rng.random(B) < 0.3] = msb * bs
    cu = np.concatenate([[0], np.cumsum(qo)]).astype(np.int64)
    tq = int(cu[-1])
    q = rng.standard_normal((tq, hq, d)).astype(np.float32)
    k = rng.standard_normal((num_pages, hkv, ps, d)).astype(np.float32)
    v = rng.standard_normal((num_pages, hkv, ps, d)).astype(np.float32)
    if bf16:
        from inputs import bf16_bits
        k, v = bf16_bits(k), bf16_bits(v)
    if full:
        sel = full_selection(tq, hkv, msb, rng, pad=int(rng.integers(0, 3)))
    else:
        topk = int(rng.integers(1, msb + 2))
        sel = rng.integers(-1, msb, size=(tq, hkv, topk)).astype(np.int32)
    return dict(q=q, k=k, v=v, bt=perm, cu=cu, used=lens if pass_used else None, sel=sel,
                hq=hq, hkv=hkv, d=d, bs=bs, ps=ps, scale=float(np.float32(1.0 / math.sqrt(d))),
                msb=msb)


def _run_sparse(c, causal, L):
    out, lse, idx, parts = oracle.attention(c["q"], c["k"], c["v"], c["sel"], c["bt"], c["cu"],
                                            c["used"], c["hq"], c["d"], c["bs"], c["ps"],
                                            c["scale"], causal, _lib=L)
    dout, dlse = oracle.direct(c["q"], c["k"], c["v"], c["sel"], c["bt"], c["cu"], c["used"],
                               c["hq"], c["d"], c["bs"], c["ps"], c["scale"], causal, _lib=L)
    return out, lse, dout, dlse, idx, parts


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: infinities differ"
    err = np.max(np.abs(a[fin] - b[fin]), initial=0.0)
    scale = max(np.max(np.abs(b[fin]), initial=0.0), 1.0)
    assert err <= tol * scale, f"{what}: max err {err:.3e} > {tol:.1e}"


def _vs_dense(c, causal, L, what):
    out, lse, dout, dlse, _, _ = _run_sparse(c, causal, L)
    ref, rlse = dense_reference(c["q"], c["k"], c["v"], c["bt"], c["cu"], c["used"], c["hkv"],
                                c["d"], c["bs"], c["ps"], c["scale"], causal)
    _close(out, ref, 1e-12, f"{what}: combine(partials) vs dense")
    _close(lse, rlse, 1e-12, f"{what}: lse vs dense")
    _close(dout, ref, 1e-12, f"{what}: direct vs dense")
    _close(dlse, rlse, 1e-12, f"{what}: direct lse vs dense")


# --------------------------------------------------------------------------- pins


def pin_types(L):
    g = json.load(open(os.path.join(GOLDEN, "types_fixtures.json")))
    s = g["selection_row_major"]
    for i, h, r, val in s["expect"]:
        assert oracle.selection_get(s["flat"], s["hkv"], s["topk"], i, h, r, _lib=L) == val
    for case in g["cu_seqlens_invalid"]["cases"]:
        assert oracle.validate_cu_seqlens(case, _lib=L) == "CU_SEQLENS", case
    v = g["cu_seqlens_valid"]
    assert oracle.validate_cu_seqlens(v["prefix"], _lib=L) == "OK"
    for i, b in g["batch_of"]["expect"]:
        assert oracle.batch_of(g["batch_of"]["prefix"], i, _lib=L) == b, (i, b)


def pin_dense_fixtures(L):
    for make in (fixture_f1, fixture_f2):
        c = make()
        for causal in (False, True):
            _vs_dense(c, causal, L, f"{make.__name__} causal={causal}")


def pin_dense_random(L, seeds=range(40)):
    for s in seeds:
        for causal in (False, True, 2):
            c = random_case(s, bf16=(s % 3 == 0), pass_used=(s % 4 != 1))
            _vs_dense(c, causal, L, f"random seed={s} causal={causal}")


def pin_causal_modes(L, seeds=range(12)):
    """Left- and right-aligned limits coincide when every sequence's KV length
    equals its query count (lk - qo + t = t), and differ otherwise; the
    left-aligned first query of a chunk sees the block holding position 0
    only through that one key."""
    for s in seeds:
        c = random_case(s, allow_empty_seq=False)
        rng = np.random.default_rng(100 + s)
        lens = rng.integers(1, c["msb"] * c["bs"] + 1, size=len(c["cu"]) - 1)
        c["used"] = lens.astype(np.int32)                  # lk_b = qo_b
        c["cu"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        tq = int(c["cu"][-1])
        c["q"] = rng.standard_normal((tq, c["hq"], c["d"])).astype(np.float32)
        c["sel"] = full_selection(tq, c["hkv"], c["msb"])
        o1, l1, _, _, _, _ = _run_sparse(c, 1, L)
        o2, l2, _, _, _, _ = _run_sparse(c, 2, L)
        _close(o1, o2, 0.0, f"seed {s}: modes agree when lk == qo")
        _close(l1, l2, 0.0, f"seed {s}: lse")
    c = fixture_f1()
    o1, _, _, _, _, _ = _run_sparse(c, 1, L)
    o2, _, _, _, _, _ = _run_sparse(c, 2, L)
    assert not np.allclose(o1, o2), "left-aligned equals right-aligned on a chunk with lk > qo"


def pin_invariance(L, seeds=range(12)):
    """Permuting ranks and adding -1 padding leaves out/lse unchanged."""
    for s in seeds:
        rng = np.random.default_rng(1000 + s)
        c = random_case(s, full=False)
        causal = bool(s % 2)
        out, lse, *_ = _run_sparse(c, causal, L)
        sel = c["sel"]
        tq, hkv, topk = sel.shape
        pad = np.full((tq, hkv, 3), -1, np.int32)
        sel2 = np.concatenate([sel, pad], axis=2)
        for i in range(tq):
            for h in range(hkv):
                sel2[i, h] = rng.permutation(sel2[i, h])
        c2 = dict(c, sel=sel2)
        out2, lse2, *_ = _run_sparse(c2, causal, L)
        _close(out2, out, 1e-12, f"invariance seed={s}")
        _close(lse2, lse, 1e-12, f"invariance lse seed={s}")


def pin_single_block(L, seeds=range(10)):
    """One selected block: plain softmax attention over that block's keys."""
    for s in seeds:
        rng = np.random.default_rng(2000 + s)
        c = random_case(s, holes=False, allow_empty_seq=False)
        tq, hkv = c["q"].shape[0], c["hkv"]
        msb = c["msb"]
        blk = rng.integers(0, msb, size=(tq, hkv, 1)).astype(np.int32)
        c["sel"] = blk
        out, lse, dout, _, _, _ = _run_sparse(c, False, L)
        qhead = c["hq"] // hkv
        for b in range(len(c["cu"]) - 1):
            lk = msb * c["bs"] if c["used"] is None else max(int(c["used"][b]), 0)
            for i in range(int(c["cu"][b]), int(c["cu"][b + 1])):
                for h in range(hkv):
                    bk = int(blk[i, h, 0])
                    keys = [p for p in range(bk * c["bs"], min((bk + 1) * c["bs"], lk))]
                    for qh in range(qhead):
                        hq = h * qhead + qh
                        if not keys:
                            assert np.all(out[i, hq] == 0) and lse[i, hq] == -np.inf
                            continue
                        K = np.array([oracle_free_f64(c["k"])[c["bt"][b, p // c["ps"]], h,
                                                             p % c["ps"]] for p in keys])
                        V = np.array([oracle_free_f64(c["v"])[c["bt"][b, p // c["ps"]], h,
                                                             p % c["ps"]] for p in keys])
                        sc = c["scale"] * (K @ c["q"][i, hq].astype(np.float64))
                        w = np.exp(sc - sc.max())
                        ref = (w @ V) / w.sum()
                        _close(out[i, hq], ref, 1e-12, f"single block seed={s}")


def pin_equal_keys(L):
    """All keys equal: softmax weights are uniform, out = mean of selected V."""
    rng = np.random.default_rng(7)
    c = random_case(3, holes=False, full=False, allow_empty_seq=False)
    c["k"] = np.broadcast_to(rng.standard_normal(c["d"]).astype(np.float32),
                             c["k"].shape).copy()
    out, _, _, _, idx, _ = _run_sparse(c, False, L)
    vf = oracle_free_f64(c["v"])
    qhead = c["hq"] // c["hkv"]
    msb = idx["msb"]
    for b in range(len(c["cu"]) - 1):
        lk = msb * c["bs"] if c["used"] is None else max(int(c["used"][b]), 0)
        for i in range(int(c["cu"][b]), int(c["cu"][b + 1])):
            for h in range(c["hkv"]):
                rows = []
                for blk in c["sel"][i, h]:
                    if blk < 0 or blk * c["bs"] >= lk:
                        continue
                    for p in range(blk * c["bs"], min((blk + 1) * c["bs"], lk)):
                        page = c["bt"][b, p // c["ps"]]
                        if page >= 0:
                            rows.append(vf[page, h, p % c["ps"]])
                for qh in range(qhead):
                    ref = np.mean(rows, axis=0) if rows else np.zeros(c["d"])
                    _close(out[i, h * qhead + qh], ref, 1e-12, "equal keys")


def pin_partials(L, seeds=range(10)):
    """1 <= l <= keys; o / l lies in the box of the block's V rows; a block
    with one key gives o = v, l = 1 and m = scale * <q, k>."""
    for s in seeds:
        c = random_case(s, full=False, allow_empty_seq=False)
        _, _, _, _, idx, (o, m, l) = _run_sparse(c, bool(s % 2), L)
        qhead = c["hq"] // c["hkv"]
        bs = c["bs"]
        live = l > 0
        assert np.all(l[live] >= 1.0 - 1e-12) and np.all(l[live] <= bs + 1e-12)
        assert np.all(np.isneginf(m[~live])) and np.all(o[~live] == 0)
        vf = oracle_free_f64(c["v"])
        for h in range(c["hkv"]):
            for j in range(int(idx["num_sel"][h])):
                raw = int(idx["sel_slots"][h, j])
                b, blk = divmod(raw, idx["msb"])
                lk = idx["msb"] * bs if c["used"] is None else max(int(c["used"][b]), 0)
                rows = [vf[c["bt"][b, p // c["ps"]], h, p % c["ps"]]
                        for p in range(blk * bs, min((blk + 1) * bs, lk))
                        if c["bt"][b, p // c["ps"]] >= 0]
                e0 = idx["edge_head_base"][h] + idx["sel_offsets"][h, j]
                e1 = idx["edge_head_base"][h] + idx["sel_offsets"][h, j + 1]
                for e in range(e0, e1):
                    for qh in range(qhead):
                        r = e * qhead + qh
                        if l[r] == 0:
                            continue
                        lo = np.min(rows, axis=0) - 1e-12
                        hi = np.max(rows, axis=0) + 1e-12
                        ratio = o[r] / l[r]
                        assert np.all(ratio >= lo) and np.all(ratio <= hi), "convex hull"
    # one key per block
    c = fixture_f1()
    c["used"] = np.array([5], np.int32)      # the last block [4, 6) keeps one key
    _, _, _, _, idx, (o, m, l) = _run_sparse(c, False, L)
    j = list(idx["sel_slots"][0, : idx["num_sel"][0]]).index(2)
    e = idx["sel_offsets"][0, j]
    vf = oracle_free_f64(c["v"])
    kf = oracle_free_f64(c["k"])
    for edge in range(e, idx["sel_offsets"][0, j + 1]):
        qi = idx["edges"][edge, 0]
        assert l[edge] == 1.0
        assert np.allclose(o[edge], vf[2, 0, 0], rtol=0, atol=0)
        assert abs(m[edge] - c["scale"] * float(kf[2, 0, 0] @ c["q"][qi, 0])) < 1e-12


def brute_force_index(sel, cu, used, max_pages, bs, ps, split_edges=0):
    """The index built by sorting every kept (query, rank) entry by
    (kv head, raw slot, query, rank): a different construction from the
    oracle's bucket append."""
    tq, hkv, topk = sel.shape
    B = len(cu) - 1
    msb = max_pages // (bs // ps)
    nbs = B * msb
    entries = []
    inv = np.full((hkv, tq, topk), -1, np.int64)
    for i in range(tq):
        b = int(np.searchsorted(cu, i, side="right") - 1)
        lk = msb * bs if used is None else max(int(used[b]), 0)
        for h in range(hkv):
            for r in range(topk):
                s = int(sel[i, h, r])
                if s >= 0 and s * bs < lk:
                    entries.append((h, b * msb + s, i, r))
    entries.sort()
    sel_slots = np.full((hkv, nbs), -1, np.int64)
    sel_offsets = np.zeros((hkv, nbs + 1), np.int64)
    num_sel = np.zeros(hkv, np.int64)
    ehb = np.zeros(hkv + 1, np.int64)
    edges = np.array([(i, r) for (_, _, i, r) in entries], np.int64).reshape(-1, 2)
    splits = []
    for h in range(hkv):
        mine = [(n, e) for n, e in enumerate(entries) if e[0] == h]
        ehb[h + 1] = ehb[h] + len(mine)
        slots = sorted({e[1] for _, e in mine})
        num_sel[h] = len(slots)
        for j, slot in enumerate(slots):
            sel_slots[h, j] = slot
            first = min(n for n, e in mine if e[1] == slot)
            sel_offsets[h, j] = first - ehb[h]
        sel_offsets[h, len(slots):] = len(mine)
        for n, (hh, slot, i, r) in mine:
            inv[h, i, r] = n - ehb[h]
        for j in range(len(slots)):
            a = ehb[h] + sel_offsets[h, j]
            z = ehb[h] + sel_offsets[h, j + 1]
            step = split_edges if split_edges > 0 else z - a
            for s0 in range(a, z, step):
                splits.append((h, j, s0, min(s0 + step, z)))
    return dict(sel_slots=sel_slots, sel_offsets=sel_offsets, num_sel=num_sel,
                edge_head_base=ehb, edges=edges, inv=inv,
                splits=np.array(splits, np.int64).reshape(-1, 4))


INDEX_KEYS = ("sel_slots", "sel_offsets", "num_sel", "edge_head_base", "edges", "inv", "splits")


def pin_index_bruteforce(L, seeds=range(60)):
    for s in seeds:
        rng = np.random.default_rng(3000 + s)
        c = random_case(s, full=bool(s % 2 == 0))
        sel = c["sel"]
        if s % 5 == 0 and sel.shape[2] > 1:
            sel[..., 1] = sel[..., 0]            # a block repeated at two ranks
        split = int(rng.integers(0, 4))
        got = oracle.build_index(sel, c["cu"], c["used"], c["bt"].shape[1], c["bs"], c["ps"],
                                 split, _lib=L)
        ref = brute_force_index(sel, c["cu"], c["used"], c["bt"].shape[1], c["bs"], c["ps"],
                                split)
        for key in INDEX_KEYS:
            assert np.array_equal(np.asarray(got[key], np.int64), ref[key]), \
                f"index seed={s}: {key} differs"


def pin_errors(L):
    c = fixture_f2()
    args = (c["cu"], c["used"], 3, c["bs"], c["ps"])

    def kind(fn):
        try:
            fn()
        except oracle.OracleError as e:
            return e.kind
        return "OK"

    sel = c["sel"].copy()
    assert kind(lambda: oracle.build_index(sel, *args, _lib=L)) == "OK"
    bad = sel.copy(); bad[1, 0, 2] = 3                        # == msb
    assert kind(lambda: oracle.build_index(bad, *args, _lib=L)) == "SELECTED_RANGE"
    bad = sel.copy(); bad[0, 1, 0] = -2
    assert kind(lambda: oracle.build_index(bad, *args, _lib=L)) == "SELECTED_RANGE"
    assert kind(lambda: oracle.build_index(sel, c["cu"], c["used"], 3, 6, 4, _lib=L)) == \
        "BLOCK_PAGE"
    assert kind(lambda: oracle.build_index(sel[:0], np.array([0, 0, 0]), c["used"], 3, 4, 4,
                                           _lib=L)) == "EMPTY"
    assert kind(lambda: oracle.build_index(sel, np.array([0, 2, 1, 3]), c["used"], 3, 4, 4,
                                           _lib=L)) == "CU_SEQLENS"
    assert kind(lambda: oracle.build_index(sel, np.array([0, 2, 4]), c["used"], 3, 4, 4,
                                           _lib=L)) == "SHAPE"
    idx = oracle.build_index(sel, *args, _lib=L)
    assert kind(lambda: oracle.forward(c["q"], c["k"], c["v"], idx, c["bt"], c["cu"], c["used"],
                                       3, c["d"], c["scale"], False, _lib=L)) == "HEAD_COUNT"
    bt = c["bt"].copy(); bt[1, 2] = 3                          # page id == num_pages
    assert kind(lambda: oracle.forward(c["q"], c["k"], c["v"], idx, bt, c["cu"], c["used"],
                                       c["hq"], c["d"], c["scale"], False, _lib=L)) == "SHAPE"
    # All padding: no edges, not an error; the output is zero, lse -inf.
    allpad = np.full_like(sel, -1)
    out, lse, idx0, _ = oracle.attention(c["q"], c["k"], c["v"], allpad, c["bt"], c["cu"],
                                         c["used"], c["hq"], c["d"], c["bs"], c["ps"],
                                         c["scale"], False, _lib=L)
    assert idx0["edges"].shape[0] == 0 and np.all(out == 0) and np.all(np.isneginf(lse))


def pin_round_bf16(L):
    """Nearest-bfloat16 rounding against the library conversion float32 ->
    bfloat16 (round to nearest even) on normal, subnormal, huge and tie
    values, plus hand-checked ties and limits."""
    import torch
    rng = np.random.default_rng(7)
    x = rng.standard_normal(20000).astype(np.float32)
    ties = np.float32([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -133 * 1.5,
                       2 ** -133 * 0.5, 2 ** -126 * (1 + 2 ** -8), 3.3895313892515355e38])
    with np.errstate(over="ignore"):
        x = np.concatenate([x, x * np.float32(1e-39), x * np.float32(1e36), ties])
    got = oracle.round_bf16(x.astype(np.float64), _lib=L)
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, lib), "bf16 rounding differs from the library conversion"
    # ties go to the even neighbour; the subnormal grid is 2^-133; the largest
    # bf16 value stays, the next grid point overflows
    r = lambda v: float(oracle.round_bf16(np.float64([v]), _lib=L)[0])
    assert r(1 + 2 ** -8) == 1.0 and r(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    assert r(2 ** -133 * 1.5) == 2 ** -132 and r(2 ** -133 * 0.5) == 0.0
    assert r((2 - 2 ** -7) * 2.0 ** 127) == (2 - 2 ** -7) * 2.0 ** 127
    assert r((2 - 2 ** -8) * 2.0 ** 127) == np.inf
    assert r(1.0 / 3.0) == 0.333984375


def pin_bf16_partials(L, seeds=range(8)):
    """16-bit o partials: each combined output moves from the f32-partial one
    by at most 2^-8 sum_r w_r |o_r| / L (every o value carries a relative
    rounding error of at most 2^-8), and does move; with bf16 V and blocks of
    one live key, o = v is a bfloat16 value already and nothing changes."""
    for s in seeds:
        c = random_case(s, full=False, allow_empty_seq=False)
        args = (c["q"], c["k"], c["v"], c["sel"], c["bt"], c["cu"], c["used"], c["hq"], c["d"],
                c["bs"], c["ps"], c["scale"], bool(s % 2))
        out, lse, idx, (o, m, l) = oracle.attention(*args, _lib=L)
        out16, lse16, _, (o16, m16, l16) = oracle.attention(*args, partial_dtype="bf16", _lib=L)
        assert np.array_equal(m, m16) and np.array_equal(l, l16) and np.array_equal(lse, lse16)
        qhead = c["hq"] // c["hkv"]
        bound = np.zeros_like(out)
        for h in range(c["hkv"]):
            for i in range(idx["tq"]):
                for qh in range(qhead):
                    rows = [(idx["edge_head_base"][h] + p) * qhead + qh
                            for p in idx["inv"][h, i] if p >= 0]
                    rows = [r for r in rows if np.isfinite(m[r])]
                    if not rows:
                        continue
                    mm = max(m[r] for r in rows)
                    w = [np.exp(m[r] - mm) for r in rows]
                    big_l = sum(wi * l[r] for wi, r in zip(w, rows))
                    bound[i, h * qhead + qh] = sum(wi * np.abs(o[r]) for wi, r in
                                                   zip(w, rows)) / big_l
        diff = np.abs(out16 - out)
        assert np.all(diff <= 2.0 ** -8 * bound * (1 + 1e-9) + 1e-300), "bf16 partial bound"
        assert np.any(diff > 0), "o partials were not rounded"
    # bf16 V, one live key per block: o = v exactly, so nothing changes
    c = random_case(3, bf16=True, full=False, allow_empty_seq=False)
    c["bs"], c["ps"] = 1, 1
    c["bt"] = np.arange(c["bt"].shape[0] * c["bt"].shape[1], dtype=np.int32).reshape(
        c["bt"].shape) % (c["k"].shape[0])
    msb = c["bt"].shape[1]
    c["used"] = np.full(len(c["cu"]) - 1, msb, np.int32)
    c["sel"] = np.random.default_rng(3).integers(-1, msb, size=c["sel"].shape).astype(np.int32)
    args = (c["q"], c["k"], c["v"], c["sel"], c["bt"], c["cu"], c["used"], c["hq"], c["d"],
            c["bs"], c["ps"], c["scale"], False)
    out, _, _, (o, _, _) = oracle.attention(*args, _lib=L)
    out16, _, _, (o16, _, _) = oracle.attention(*args, partial_dtype="bf16", _lib=L)
    assert np.array_equal(o, o16) and np.array_equal(out, out16)


ALL_PINS = [pin_types, pin_dense_fixtures, pin_dense_random, pin_invariance, pin_single_block,
            pin_equal_keys, pin_partials, pin_index_bruteforce, pin_errors, pin_round_bf16,
            pin_bf16_partials, pin_causal_modes]
