"""Seeded synthetic inputs for KV-outer block-sparse paged attention.

This module holds input generation only (no attention arithmetic).  Both the
oracle-based tests and the CUDA library's callers (tests, bench) draw their
inputs from here, so that the two sides always see bit-identical data.

Values (q, k_pages, v_pages) come from a counter-based generator: element
``idx`` of tensor ``stream`` under ``seed`` is a function of (seed, stream,
idx) alone, so any slice of a 70 GB pool can be produced on the host without
the rest, and the device fill kernel (``fill.cu``) produces the same bits:

    key   = seed * 16 + stream                              (uint64)
    x     = idx + key * 0xD1B54A32D192ED03                   (mod 2**64)
    z     = splitmix64 finaliser of x (Steele, Lea & Flood, 2014)
    u     = sum of the four 16-bit fields of z               (0 .. 262140)
    value = float32(u - 131070) * float32(1 / sqrt((65536**2 - 1) / 3))

``u`` is an Irwin-Hall sum of four discrete uniforms, so ``value`` has mean 0
and variance 1 (an approximation of N(0, 1) bounded by |x| < 3.47).  The int
to float conversion is exact and the one multiply is rounded to nearest, so
numpy and CUDA agree bit for bit.  bf16 pools take the round-to-nearest-even
bf16 of that float.

Selections, block tables and sequence lengths come from numpy's PCG64 seeded
with (seed, workload id); their structure follows the five serving workloads
described in the design notes (tiny, GQA decode, chunked prefill, skewed
selection, long-context decode).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

STREAM_Q = 1
STREAM_K = 2
STREAM_V = 3

_MUL_KEY = np.uint64(0xD1B54A32D192ED03)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_IH_CENTER = 131070
_IH_SCALE = np.float32(1.0 / math.sqrt((65536.0 ** 2 - 1.0) / 3.0))


def _splitmix64(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def counter_normal(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """float32 values of elements [start, start+count) of tensor `stream`."""
    return counter_normal_at(seed, stream, np.arange(start, start + count, dtype=np.uint64))


def counter_normal_at(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """float32 values of the elements with flat indices `idx` of tensor `stream`."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        key = np.uint64(seed * 16 + stream)
        z = _splitmix64(idx + key * _MUL_KEY)
    mask = np.uint64(0xFFFF)
    u = ((z & mask) + ((z >> np.uint64(16)) & mask) + ((z >> np.uint64(32)) & mask)
         + ((z >> np.uint64(48)) & mask)).astype(np.int64)
    return (u - _IH_CENTER).astype(np.float32) * _IH_SCALE


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even bf16 bit patterns (uint16) of finite float32 values."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- workloads


@dataclass
class Workload:
    """One synthetic problem: geometry, host index inputs and value seeds."""

    name: str
    seed: int
    batch: int
    qo_lens: np.ndarray          # [B] queries per sequence
    used_kv_lens: np.ndarray     # [B] int32
    hq: int
    hkv: int
    head_dim: int
    page_size: int
    block_size: int
    max_pages: int
    topk: int
    causal: bool
    kv_dtype: str                # "f32" or "bf16"
    selected: np.ndarray         # [tq, hkv, topk] int32
    block_tables: np.ndarray     # [B, max_pages] int32
    num_pages: int
    softmax_scale: float
    pass_used: bool = True       # False: call with used_kv_lens = None
    notes: dict = field(default_factory=dict)

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.qo_lens)]).astype(np.int64)

    @property
    def tq(self) -> int:
        return int(np.sum(self.qo_lens))

    @property
    def qhead(self) -> int:
        return self.hq // self.hkv

    @property
    def ppb(self) -> int:
        return self.block_size // self.page_size

    @property
    def msb(self) -> int:
        return self.max_pages // self.ppb

    @property
    def used(self):
        return self.used_kv_lens if self.pass_used else None

    @property
    def page_elems(self) -> int:
        return self.hkv * self.page_size * self.head_dim

    # ---- values on the host

    def q_host(self) -> np.ndarray:
        n = self.tq * self.hq * self.head_dim
        return counter_normal(self.seed, STREAM_Q, 0, n).reshape(self.tq, self.hq, self.head_dim)

    def _pool_host(self, stream: int, page_ids=None):
        pe = self.page_elems
        if page_ids is None:
            vals = counter_normal(self.seed, stream, 0, self.num_pages * pe)
            shape = (self.num_pages, self.hkv, self.page_size, self.head_dim)
        else:
            page_ids = np.asarray(page_ids, dtype=np.int64)
            vals = np.concatenate([counter_normal(self.seed, stream, int(p) * pe, pe)
                                   for p in page_ids]) if page_ids.size else np.zeros(0, np.float32)
            shape = (page_ids.size, self.hkv, self.page_size, self.head_dim)
        vals = vals.reshape(shape)
        if self.kv_dtype == "bf16":
            return bf16_bits(vals)
        return vals

    def k_host(self, page_ids=None):
        """K pool (or the listed pages) as float32, or bf16 bits (uint16)."""
        return self._pool_host(STREAM_K, page_ids)

    def v_host(self, page_ids=None):
        return self._pool_host(STREAM_V, page_ids)

    def compact_pool(self, queries=None):
        """Only the pages the given queries' kept blocks touch, with a block
        table remapped onto them: (k, v, block_tables, num_pages)."""
        sel = self.selected if queries is None else self.selected[np.asarray(queries)]
        cu = self.cu_seqlens_q
        qs = np.arange(self.tq) if queries is None else np.asarray(queries)
        bt = self.block_tables
        needed = set()
        for row, i in enumerate(qs):
            b = int(np.searchsorted(cu, i, side="right") - 1)
            lk = max(int(self.used_kv_lens[b]), 0) if self.pass_used else self.msb * self.block_size
            for blk in np.unique(sel[row]):
                if blk < 0 or blk * self.block_size >= lk:
                    continue
                for p in range(self.ppb):
                    page = int(bt[b, blk * self.ppb + p])
                    if page >= 0:
                        needed.add(page)
        ids = np.array(sorted(needed), dtype=np.int64)
        remap = np.full(self.num_pages, -1, np.int32)
        remap[ids] = np.arange(ids.size, dtype=np.int32)
        bt2 = np.where(bt >= 0, remap[np.clip(bt, 0, None)], -1).astype(np.int32)
        return self.k_host(ids), self.v_host(ids), bt2, max(len(ids), 1)


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.default_rng([seed, tag])


def _distinct(rng, n_rows: int, n_choices: int, k: int) -> np.ndarray:
    """k distinct uniform draws from range(n_choices) per row."""
    keys = rng.random((n_rows, n_choices))
    return np.argpartition(keys, k - 1, axis=1)[:, :k] if k < n_choices else \
        np.argsort(keys, axis=1)[:, :k]


def _tables(rng, batch: int, max_pages: int, lens=None, page_size=1, pad_tail=False):
    pool = batch * max_pages
    perm = rng.permutation(pool).astype(np.int32)
    bt = perm.reshape(batch, max_pages).copy()
    if pad_tail and lens is not None:
        for b in range(batch):
            live = -(-int(lens[b]) // page_size)
            bt[b, live:] = -1
    return bt, pool


def tiny(seed: int = 0) -> Workload:
    """B=1, 4 queries, Hq=4, Hkv=2, d=32, page 16, block 32, kv 256 (8 blocks),
    topk=2 distinct uniform blocks, non-causal, f32."""
    rng = _rng(seed, 0)
    B, qo, hq, hkv, d, ps, bs, kv, topk = 1, 4, 4, 2, 32, 16, 32, 256, 2
    max_pages = kv // ps
    sel = _distinct(rng, qo * hkv, kv // bs, topk).reshape(qo, hkv, topk).astype(np.int32)
    bt, pool = _tables(rng, B, max_pages)
    return Workload("tiny", seed, B, np.array([qo]), np.array([kv], np.int32), hq, hkv, d, ps,
                    bs, max_pages, topk, False, "f32", sel, bt, pool, 1.0 / math.sqrt(d))


def gqa_decode(seed: int = 0, batch: int = 64, kv_min: int = 4096, kv_max: int = 32768,
               hq: int = 32, hkv: int = 8, head_dim: int = 128, page_size: int = 16,
               block_size: int = 64, topk: int = 16, kv_dtype: str = "f32") -> Workload:
    """One query per sequence; used_kv_lens uniform in [kv_min, kv_max]; rank 0
    is the sequence's last (local) block, the other topk-1 are distinct uniform
    earlier blocks; causal (right-aligned); pages randomly permuted over the
    pool, table entries past the sequence's length are -1."""
    rng = _rng(seed, 1)
    max_pages = -(-kv_max // block_size) * (block_size // page_size)
    lens = rng.integers(kv_min, kv_max + 1, size=batch).astype(np.int32)
    sel = np.empty((batch, hkv, topk), np.int32)
    for b in range(batch):
        last = -(-int(lens[b]) // block_size) - 1
        sel[b, :, 0] = last
        sel[b, :, 1:] = _distinct(rng, hkv, last, topk - 1)
    bt, pool = _tables(rng, batch, max_pages, lens, page_size, pad_tail=True)
    return Workload("gqa_decode", seed, batch, np.ones(batch, np.int64), lens, hq, hkv, head_dim,
                    page_size, block_size, max_pages, topk, True, kv_dtype, sel, bt, pool,
                    1.0 / math.sqrt(head_dim))


def chunked_prefill(seed: int = 0, batch: int = 4, qo_len: int = 2048, kv_len: int = 32768,
                    hq: int = 64, hkv: int = 8, head_dim: int = 128, page_size: int = 64,
                    block_size: int = 128, topk: int = 32, kv_dtype: str = "f32") -> Workload:
    """qo_len queries per sequence at the end of a kv_len context; rank 0 is the
    query's own (local) block, the other topk-1 are distinct uniform earlier
    blocks; causal (right-aligned)."""
    rng = _rng(seed, 2)
    max_pages = -(-kv_len // block_size) * (block_size // page_size)
    tq = batch * qo_len
    sel = np.empty((tq, hkv, topk), np.int32)
    for b in range(batch):
        for t in range(qo_len):
            i = b * qo_len + t
            local = (kv_len - qo_len + t) // block_size
            sel[i, :, 0] = local
            sel[i, :, 1:] = _distinct(rng, hkv, local, topk - 1)
    bt, pool = _tables(rng, batch, max_pages)
    lens = np.full(batch, kv_len, np.int32)
    return Workload("chunked_prefill", seed, batch, np.full(batch, qo_len, np.int64), lens, hq,
                    hkv, head_dim, page_size, block_size, max_pages, topk, True, kv_dtype, sel,
                    bt, pool, 1.0 / math.sqrt(head_dim))


def skewed(seed: int = 0, batch: int = 16, qo_len: int = 512, kv_len: int = 65536,
           hq: int = 32, hkv: int = 4, head_dim: int = 128, page_size: int = 16,
           block_size: int = 64, topk: int = 24, zipf_s: float = 1.2, pad_p: float = 0.15,
           kv_dtype: str = "f32") -> Workload:
    """topk distinct block ids per (query, kv head) drawn Zipf(zipf_s) over
    popularity ranks 1..msb without replacement (Gumbel top-k), mapped to block
    ids through a per-sequence permutation; each rank is -1 with probability
    pad_p; non-causal."""
    rng = _rng(seed, 3)
    max_pages = -(-kv_len // block_size) * (block_size // page_size)
    msb = max_pages // (block_size // page_size)
    logw = -zipf_s * np.log(np.arange(1, msb + 1, dtype=np.float64))
    tq = batch * qo_len
    sel = np.empty((tq, hkv, topk), np.int32)
    for b in range(batch):
        perm = rng.permutation(msb).astype(np.int32)
        g = -np.log(-np.log(rng.random((qo_len * hkv, msb))))
        ranks = np.argpartition(-(logw + g), topk - 1, axis=1)[:, :topk]
        sel[b * qo_len:(b + 1) * qo_len] = perm[ranks].reshape(qo_len, hkv, topk)
    pad = rng.random(sel.shape) < pad_p
    sel[pad] = -1
    bt, pool = _tables(rng, batch, max_pages)
    lens = np.full(batch, kv_len, np.int32)
    return Workload("skewed", seed, batch, np.full(batch, qo_len, np.int64), lens, hq, hkv,
                    head_dim, page_size, block_size, max_pages, topk, False, kv_dtype, sel, bt,
                    pool, 1.0 / math.sqrt(head_dim))


def long_decode(seed: int = 0, batch: int = 128, kv_min: int = 65536, kv_max: int = 131072,
                hq: int = 64, hkv: int = 8, head_dim: int = 128, page_size: int = 16,
                block_size: int = 64, topk: int = 64, pad_p: float = 0.10,
                kv_dtype: str = "bf16") -> Workload:
    """One query per sequence; used_kv_lens uniform in [kv_min, kv_max]; topk
    distinct uniform blocks of the sequence; each rank -1 with probability
    pad_p; causal (right-aligned); bf16 K/V."""
    rng = _rng(seed, 4)
    max_pages = -(-kv_max // block_size) * (block_size // page_size)
    lens = rng.integers(kv_min, kv_max + 1, size=batch).astype(np.int32)
    sel = np.empty((batch, hkv, topk), np.int32)
    for b in range(batch):
        nblk = -(-int(lens[b]) // block_size)
        sel[b] = _distinct(rng, hkv, nblk, topk)
    pad = rng.random(sel.shape) < pad_p
    sel[pad] = -1
    bt, pool = _tables(rng, batch, max_pages, lens, page_size, pad_tail=True)
    return Workload("long_decode", seed, batch, np.ones(batch, np.int64), lens, hq, hkv, head_dim,
                    page_size, block_size, max_pages, topk, True, kv_dtype, sel, bt, pool,
                    1.0 / math.sqrt(head_dim))


#: The five serving workloads at full size.
FULL = {
    "tiny": tiny,
    "gqa_decode": gqa_decode,
    "chunked_prefill": chunked_prefill,
    "chunked_prefill_bf16": lambda seed=0: replace(chunked_prefill(seed, kv_dtype="bf16"),
                                                   name="chunked_prefill_bf16"),
    "skewed": skewed,
    "long_decode": long_decode,
}


#: Reduced versions with the same structure, small enough for the oracle to
#: check every output in seconds while still covering several blocks, several
#: sequences, ragged lengths and every code path.
def small(name: str, seed: int = 0) -> Workload:
    if name == "tiny":
        return tiny(seed)
    if name == "gqa_decode":
        return gqa_decode(seed, batch=6, kv_min=1100, kv_max=2000, topk=8)
    if name == "chunked_prefill":
        return chunked_prefill(seed, batch=2, qo_len=40, kv_len=1000, hq=16, hkv=2, topk=6)
    if name == "chunked_prefill_bf16":
        w = chunked_prefill(seed, batch=2, qo_len=40, kv_len=1000, hq=16, hkv=2, topk=6,
                            kv_dtype="bf16")
        return replace(w, name="chunked_prefill_bf16")
    if name == "skewed":
        return skewed(seed, batch=3, qo_len=48, kv_len=2048, topk=10)
    if name == "long_decode":
        return long_decode(seed, batch=5, kv_min=1500, kv_max=4000, topk=12)
    raise KeyError(name)


# --------------------------------------------------------------------------- device fill

_HERE = os.path.dirname(os.path.abspath(__file__))
_FILL_SRC = os.path.join(_HERE, "fill.cu")
_FILL_LIB = os.path.join(_HERE, "_build", "libsa_inputs.so")
_fill_lock = threading.Lock()
_fill = None


def build_fill(nvcc: str = "nvcc") -> str:
    """Compile the device fill kernel (sm_103a) into inputs/_build/."""
    os.makedirs(os.path.dirname(_FILL_LIB), exist_ok=True)
    tmp = _FILL_LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-O3", "-shared", "-Xcompiler", "-fPIC",
                    "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, _FILL_SRC],
                   check=True)
    os.replace(tmp, _FILL_LIB)
    return _FILL_LIB


def _fill_lib():
    global _fill
    with _fill_lock:
        if _fill is None:
            if not os.path.exists(_FILL_LIB):
                raise RuntimeError("inputs/_build/libsa_inputs.so is missing: run build()")
            lib = ctypes.CDLL(_FILL_LIB)
            lib.sa_inputs_fill.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                                           ctypes.c_void_p]
            lib.sa_inputs_fill.restype = ctypes.c_int
            _fill = lib
    return _fill


def fill_device(tensor, seed: int, stream_id: int, start: int = 0, bf16: bool = False,
                cuda_stream=None) -> None:
    """Fill a contiguous CUDA tensor (float32, or int16/bfloat16 storage when
    bf16) with elements [start, start + numel) of the counter generator."""
    import torch

    s = cuda_stream if cuda_stream is not None else torch.cuda.current_stream(tensor.device)
    rc = _fill_lib().sa_inputs_fill(ctypes.c_void_p(tensor.data_ptr()), tensor.numel(), start,
                                    seed, stream_id, int(bf16), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"sa_inputs_fill failed with CUDA error {rc}")


def device_tensors(w: Workload, device="cuda"):
    """q, k_pages, v_pages on the device, filled by the counter generator."""
    import torch

    q = torch.empty((w.tq, w.hq, w.head_dim), dtype=torch.float32, device=device)
    fill_device(q, w.seed, STREAM_Q)
    kv_t = torch.bfloat16 if w.kv_dtype == "bf16" else torch.float32
    shape = (w.num_pages, w.hkv, w.page_size, w.head_dim)
    k = torch.empty(shape, dtype=kv_t, device=device)
    v = torch.empty(shape, dtype=kv_t, device=device)
    fill_device(k, w.seed, STREAM_K, bf16=w.kv_dtype == "bf16")
    fill_device(v, w.seed, STREAM_V, bf16=w.kv_dtype == "bf16")
    return q, k, v
