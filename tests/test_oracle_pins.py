"""The oracle against the pages' printed fixtures, dense attention, the
method's invariances and closed forms (CPU only)."""
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest

import _pins
import oracle


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc.lib())


def test_direct_equals_combined_partials(orc):
    """The query-outer attention and index -> partials -> combine agree on
    arbitrary (partial, padded, repeated) selections."""
    for s in range(30):
        c = _pins.random_case(s, bf16=bool(s % 2), full=False)
        for causal in (False, True):
            out, lse, dout, dlse, _, _ = _pins._run_sparse(c, causal, orc.lib())
            _pins._close(out, dout, 1e-12, f"seed {s}")
            _pins._close(lse, dlse, 1e-12, f"seed {s} lse")


# Plausible mistakes, each planted in a private copy of the oracle source; the
# pins must reject every one of them.
MUTATIONS = [
    ("causal off by one", "pos[t] > limit", "pos[t] >= limit"),
    ("causal not right-aligned", "return lk - qo_len + q_local;", "return q_local;"),
    ("scale dropped", "score[t] = (double)softmax_scale * dot;", "score[t] = dot;"),
    ("GQA lane mapping", "int64_t hq_abs = h * qhead + qh;", "int64_t hq_abs = qh * hkv + h;"),
    ("K used for V", "o[d] += p * kv_value(v_pages", "o[d] += p * kv_value(k_pages"),
    ("max not subtracted in partials", "double p = exp(score[t] - m);\n                        l += p;\n                        int64_t base = page[t] * page_stride + (h * page_size + row[t]) * head_dim;\n                        for (int64_t d = 0; d < head_dim; ++d)\n                            o[d] += p * kv_value(v_pages, kv_is_bf16, base + d);\n                    }\n                    m_partial",
     "double p = exp(score[t]);\n                        l += p;\n                        int64_t base = page[t] * page_stride + (h * page_size + row[t]) * head_dim;\n                        for (int64_t d = 0; d < head_dim; ++d)\n                            o[d] += p * kv_value(v_pages, kv_is_bf16, base + d);\n                    }\n                    m_partial"),
    ("combine weight missing on l", "big_l += w * l_partial[row];", "big_l += l_partial[row];"),
    ("combine lane dropped", "int64_t row = (edge_head_base[h] + p) * qhead + qh;",
     "int64_t row = (edge_head_base[h] + p) * qhead;"),
    ("combine not normalised", "o[d] /= big_l;\n            lse", "(void)0;\n            lse"),
    ("drop rule boundary", "if (blk < 0 || (int64_t)blk * block_size >= lk)",
     "if (blk < 0 || (int64_t)blk * block_size > lk)"),
    ("inv absolute", "inv[inv_at] = (int32_t)pos;", "inv[inv_at] = (int32_t)(head_base + pos);"),
    ("page index ignores pages_per_block",
     "block_tables[b * max_pages + blk * ppb + page_local]",
     "block_tables[b * max_pages + blk + page_local]"),
    ("batch_of boundary", "if (prefix[i] > query)", "if (prefix[i] >= query)"),
    ("cu_seqlens rejects empty sequences", "if (prefix[i] < prefix[i - 1])",
     "if (prefix[i] <= prefix[i - 1])"),
    ("plateau skips its first entry", "for (int64_t p = j; p <= nbs; ++p)",
     "for (int64_t p = j + 1; p <= nbs; ++p)"),
    ("head base not accumulated", "head_base += running;", "head_base = running;"),
    ("selection layout transposed", "return selected[(tq_idx * hkv + hkv_idx) * topk + rank];",
     "return selected[(hkv_idx * hkv + tq_idx) * topk + rank];"),
    ("slots compacted in descending order", "for (int64_t slot = 0; slot < nbs; ++slot)",
     "for (int64_t slot = nbs - 1; slot >= 0; --slot)"),
    ("lse uses natural log of max only", "lse[i * hq + hq_abs] = big_m + log(big_l);",
     "lse[i * hq + hq_abs] = big_m;"),
    ("bf16 rounding truncates", "double y = ldexp(rint(ldexp(x, -step)), step);",
     "double y = ldexp(trunc(ldexp(x, -step)), step);"),
    ("bf16 grid one bit too fine", "int step = k - 8;", "int step = k - 9;"),
    ("left-aligned limit taken right-aligned", "    if (mode == 2)\n        return q_local;",
     "    if (mode == 2)\n        return lk - qo_len + q_local;"),
    ("bf16 subnormal grid too coarse", "if (step < -133)\n        step = -133;",
     "if (step < -126)\n        step = -126;"),
]


_RUN_PINS = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import _pins, oracle
L = oracle.load_library({so!r})
caught = []
for pin in _pins.ALL_PINS:
    try:
        pin(L)
    except (AssertionError, oracle.OracleError, ValueError, IndexError):
        caught.append(pin.__name__)
print("CAUGHT", ",".join(caught))
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(orc, name, old, new):
    """Each mutant runs in its own process: a mistake that corrupts memory
    (and so kills the process) counts as rejected too."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "sa_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor for '{name}' not found in the oracle"
    mutated = src.replace(old, new)
    here = os.path.dirname(os.path.abspath(__file__))
    with tempfile.TemporaryDirectory() as tmp:
        c_path = os.path.join(tmp, "mutant.c")
        so_path = os.path.join(tmp, "libmutant.so")
        open(c_path, "w").write(mutated)
        oracle.compile_library(c_path, so_path)
        script = _RUN_PINS.format(root=os.path.dirname(here), tests=here, so=so_path)
        r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                           timeout=600)
        line = [x for x in r.stdout.splitlines() if x.startswith("CAUGHT")]
        rejected = r.returncode != 0 or (line and line[-1].strip() != "CAUGHT")
        assert rejected, f"no pin rejects the planted mistake '{name}'"
