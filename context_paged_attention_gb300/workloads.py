"""Seeded synthetic inputs for striped paged attention (shared by tests and bench).

This module only draws inputs: row lengths, page tables, positions and
N(0, 1) values.  It holds none of the method's arithmetic (no placement, no
attention, no merge), so both the CUDA path and the float64 oracle can consume
its output without sharing any computation.

Recipe (fixed per named workload, seed = workload index unless overridden):

1. draw the row lengths (context lengths, and new-token counts for mixed steps)
   as inclusive uniform integers;
2. size the pool: ``ceil(1.2 * sum_b ceil(L_b / page_size)) + 1`` pages (an
   explicit count for the tiny workload); the last page is the sink page that
   padding rows point at;
3. draw a random permutation of the non-sink pages; row b takes the next
   ``ceil(L_b / page_size)`` entries as its page table (rows disjoint,
   randomly placed);
4. draw q, then k, then v as float32 N(0, 1), cast to bfloat16 with
   round-to-nearest-even (the tiny workload stays float32);
5. padding rows / padding tokens get NaN queries and NaN new keys/values.

bfloat16 arrays are carried as uint16 bit patterns.
"""

from __future__ import annotations

import math
import dataclasses
from dataclasses import dataclass, field

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite N(0, 1) draws, so no NaN/inf special-casing is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


@dataclass
class Workload:
    """One step of striped paged attention, as host arrays.

    Geometry: ``P`` stripes, logical ``page_size``, ``num_pages`` pool pages
    (last one = sink), ``num_q_heads``/``num_kv_heads``, ``head_dim`` (QK) and
    ``head_dim_v`` (PV).  ``mla``: one latent KV head whose first
    ``head_dim_v`` values are the value (``v_seq`` is None).

    Rows: ``num_rows`` rows in the bucket, the first ``num_real_rows`` real.
    Row b holds ``ctx_len[b]`` keys in the pool before the step and brings
    ``new_len[b]`` new tokens, query tokens ``qo_indptr[b]:qo_indptr[b+1]``;
    ``num_tokens`` (>= ``qo_indptr[-1]``) is the padded token count.
    ``decode``: one new token a row, attended from the pool (kv_len = ctx+1);
    otherwise the pool partial covers the context only and new tokens are
    attended apart.

    Values (raw: uint16 bf16 bits or float32):
      q      [num_tokens, Hq, D]
      k_seq  [sum_b L_b, Hkv, D]   row b's logical keys, L_b = ctx + new
      v_seq  [sum_b L_b, Hkv, Dv]  (None for MLA)
      seq_indptr [num_rows + 1]
    New tokens: ``positions[t]`` logical position of token t (-1 = padding);
    ``k_new``/``v_new`` [num_tokens, Hkv, D/Dv] (NaN for padding tokens).
    Page table (CSR): ``kv_page_indptr`` [num_rows+1], ``kv_page_indices``.
    """

    name: str
    dtype: str
    P: int
    page_size: int
    num_pages: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    head_dim_v: int
    mla: bool
    scale: float
    decode: bool
    num_rows: int
    num_real_rows: int
    num_tokens: int
    ctx_len: np.ndarray
    new_len: np.ndarray
    qo_indptr: np.ndarray
    seq_indptr: np.ndarray
    kv_page_indptr: np.ndarray
    kv_page_indices: np.ndarray
    positions: np.ndarray
    q: np.ndarray
    k_seq: np.ndarray
    v_seq: np.ndarray | None
    k_new: np.ndarray
    v_new: np.ndarray | None
    meta: dict = field(default_factory=dict)
    interleave: int = 1  # runs of this many consecutive page offsets share a partner
    kv_dtype: str = "same"  # "fp8": the pool holds E4M3 codes of K / k_descale and V / v_descale
    k_descale: float = 0.0
    v_descale: float = 0.0

    @property
    def sink_page(self) -> int:
        return self.num_pages - 1

    @property
    def kv_len(self) -> np.ndarray:
        """Keys each row's queries see in the pool (decode: incl. the new token)."""
        kv = self.ctx_len + self.new_len if self.decode else self.ctx_len.copy()
        kv = kv.astype(np.int32)
        kv[self.num_real_rows:] = 0  # padding rows own no keys (their tables point at the sink page)
        return kv

    @property
    def seq_len(self) -> np.ndarray:
        return (self.ctx_len + self.new_len).astype(np.int64)

    def kv_bytes_read(self) -> int:
        """Algorithmic K/V bytes the pool partial reads: every visible key once
        (one byte a value for FP8 pools)."""
        esz = 1 if self.kv_dtype == "fp8" else (2 if self.dtype == "bf16" else 4)
        keys = int(self.kv_len[: self.num_real_rows].astype(np.int64).sum())
        per_key = self.num_kv_heads * (self.head_dim + (0 if self.mla else self.head_dim_v)) * esz
        return keys * per_key


def interleaved(w: Workload, interleave: int) -> Workload:
    """The same step over a pool whose pages move runs of ``interleave``
    consecutive offsets to one partner; the inputs are unchanged."""
    if interleave < 1 or w.page_size % (w.P * interleave) != 0:
        raise ValueError("P * interleave must divide page_size")
    name = w.name if interleave == 1 else f"{w.name}_I{interleave}"
    return dataclasses.replace(w, interleave=interleave, name=name)


def fp8_pool(w: Workload, k_descale: float, v_descale: float) -> Workload:
    """The same step with the pool kept as FP8 E4M3 codes and per-tensor
    descales (inputs unchanged; a bf16 layer only)."""
    if w.dtype != "bf16" or w.mla:
        raise ValueError("FP8 pools are for bf16 GQA layers")  # the library refuses the rest
    return dataclasses.replace(w, kv_dtype="fp8", k_descale=float(k_descale), v_descale=float(v_descale),
                               name=f"{w.name}_fp8")


def _values(rng, shape, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return x if dtype == "fp32" else f32_to_bf16_bits(x)


def _nan_like(shape, dtype):
    if dtype == "fp32":
        return np.full(shape, np.nan, dtype=np.float32)
    return np.full(shape, BF16_NAN, dtype=np.uint16)


def build_workload(name, *, dtype, P, page_size, num_q_heads, num_kv_heads, head_dim,
                   head_dim_v=None, mla=False, scale=None, decode=True,
                   ctx_len, new_len, num_real_rows=None, num_tokens=None,
                   num_pages=None, pool_factor=1.2, padding_spans=None, seed=0,
                   rng=None) -> Workload:
    """Assemble a workload from drawn row lengths.

    ``padding_spans``: new-token counts of padding rows appended after the real
    rows (0 = span-0 padding row); their tokens are padding tokens.
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    head_dim_v = head_dim if head_dim_v is None else head_dim_v
    scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
    ctx_len = np.asarray(ctx_len, dtype=np.int64)
    new_len = np.asarray(new_len, dtype=np.int64)
    B_real = len(ctx_len) if num_real_rows is None else num_real_rows
    pad = list(padding_spans or [])
    ctx_all = np.concatenate([ctx_len, np.zeros(len(pad), np.int64)])
    new_all = np.concatenate([new_len, np.asarray(pad, np.int64)])
    B = len(ctx_all)
    L = ctx_all + new_all
    L[B_real:] = 0  # padding rows own no keys
    pages_per_row = (L + page_size - 1) // page_size
    if num_pages is None:
        num_pages = int(math.ceil(pool_factor * int(pages_per_row.sum()))) + 1
    assert int(pages_per_row.sum()) <= num_pages - 1, "pool too small"
    perm = rng.permutation(num_pages - 1).astype(np.int32)
    sink = num_pages - 1
    indptr = [0]
    indices = []
    cur = 0
    for b in range(B):
        if b < B_real:
            n = int(pages_per_row[b])
            indices.extend(perm[cur: cur + n].tolist())
            cur += n
        else:
            n = 1 if new_all[b] > 0 else 0  # padding rows with tokens point at the sink page
            indices.extend([sink] * n)
        indptr.append(len(indices))
    qo_indptr = np.concatenate([[0], np.cumsum(new_all)]).astype(np.int32)
    T_used = int(qo_indptr[-1])
    T = T_used if num_tokens is None else int(num_tokens)
    assert T >= T_used
    seq_indptr = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    kv_heads = 1 if mla else num_kv_heads
    q = _values(rng, (T, num_q_heads, head_dim), dtype)
    k_seq = _values(rng, (int(seq_indptr[-1]), kv_heads, head_dim), dtype)
    v_seq = None if mla else _values(rng, (int(seq_indptr[-1]), kv_heads, head_dim_v), dtype)
    positions = np.full((T,), -1, dtype=np.int32)
    k_new = _nan_like((T, kv_heads, head_dim), dtype)
    v_new = None if mla else _nan_like((T, kv_heads, head_dim_v), dtype)
    for b in range(B_real):
        for i in range(int(new_all[b])):
            t = int(qo_indptr[b]) + i
            pos = int(ctx_all[b]) + i
            positions[t] = pos
            k_new[t] = k_seq[seq_indptr[b] + pos]
            if v_new is not None:
                v_new[t] = v_seq[seq_indptr[b] + pos]
    # queries of padding tokens (padding rows and the tail past the last row) are NaN
    q[int(qo_indptr[B_real]):] = _nan_like(q[int(qo_indptr[B_real]):].shape, dtype)
    return Workload(
        name=name, dtype=dtype, P=P, page_size=page_size, num_pages=num_pages,
        num_q_heads=num_q_heads, num_kv_heads=kv_heads, head_dim=head_dim,
        head_dim_v=head_dim_v, mla=mla, scale=float(scale), decode=decode,
        num_rows=B, num_real_rows=B_real, num_tokens=T,
        ctx_len=ctx_all.astype(np.int32), new_len=new_all.astype(np.int32),
        qo_indptr=qo_indptr, seq_indptr=seq_indptr,
        kv_page_indptr=np.asarray(indptr, dtype=np.int32),
        kv_page_indices=np.asarray(indices, dtype=np.int32),
        positions=positions, q=q, k_seq=k_seq, v_seq=v_seq, k_new=k_new, v_new=v_new,
        meta=dict(seed=seed),
    )


def _round_up(x, m):
    return (x + m - 1) // m * m


# Named workloads: index -> (description, builder).  ``scale_down`` shrinks the
# row count and lengths for oracle-sized parity runs while keeping the geometry.

def tiny_fp32(seed=1):
    """B=2, L = {37, 100}, 4 q heads / 1 KV head, D 64, page 16, P 2, 32-page pool, fp32."""
    rng = np.random.default_rng(seed)
    L = np.array([37, 100])
    return build_workload("tiny_fp32", dtype="fp32", P=2, page_size=16, num_q_heads=4,
                          num_kv_heads=1, head_dim=64, scale=1.0 / 8.0,
                          ctx_len=L - 1, new_len=np.ones(2, np.int64), num_pages=32, rng=rng,
                          seed=seed)


def gqa_decode(seed=2, batch=64, len_lo=512, len_hi=8192, padding_spans=None):
    """GQA decode bf16: 32 q / 8 KV heads, D 128, page 16, P 4, L ~ U[512, 8192]."""
    rng = np.random.default_rng(seed)
    L = rng.integers(len_lo, len_hi, size=batch, endpoint=True)
    return build_workload("gqa_decode", dtype="bf16", P=4, page_size=16, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, ctx_len=L - 1,
                          new_len=np.ones(batch, np.int64), padding_spans=padding_spans,
                          rng=rng, seed=seed)


def gqa_decode_fp8(seed=2, batch=64, len_lo=512, len_hi=8192, padding_spans=None):
    """The GQA decode step over an FP8 E4M3 pool: per-tensor descales about
    amax / 448 of the N(0, 1) draws (k 0.0123, v 0.0137)."""
    return fp8_pool(gqa_decode(seed, batch, len_lo, len_hi, padding_spans), 0.0123, 0.0137)


def long_gqa_decode(seed=3, batch=8, len_lo=65536, len_hi=131072):
    """Long-context GQA decode bf16: 64 q / 8 KV heads, D 128, page 64, P 8, L ~ U[64k, 128k]."""
    rng = np.random.default_rng(seed)
    L = rng.integers(len_lo, len_hi, size=batch, endpoint=True)
    return build_workload("long_gqa_decode", dtype="bf16", P=8, page_size=64, num_q_heads=64,
                          num_kv_heads=8, head_dim=128, ctx_len=L - 1,
                          new_len=np.ones(batch, np.int64), rng=rng, seed=seed)


def mla_decode(seed=4, batch=32, len_lo=4096, len_hi=32768):
    """MLA decode bf16: 128 q heads over one latent head (QK 576, PV 512), page 64, P 4."""
    rng = np.random.default_rng(seed)
    L = rng.integers(len_lo, len_hi, size=batch, endpoint=True)
    return build_workload("mla_decode", dtype="bf16", P=4, page_size=64, num_q_heads=128,
                          num_kv_heads=1, head_dim=576, head_dim_v=512, mla=True,
                          scale=1.0 / math.sqrt(192.0), ctx_len=L - 1,
                          new_len=np.ones(batch, np.int64), rng=rng, seed=seed)


def mixed_step(seed=5, n_decode=48, n_extend=16, dec_ctx=(1024, 16384), ext_new=(2, 256),
               ext_ctx=(0, 8192), padding_spans=None, token_multiple=256):
    """Mixed step bf16 GQA 32/8, D 128, page 16, P 4: decode rows + extend rows.

    Decode rows come first (one new token, context ~ U[dec_ctx]), then extend
    rows (new ~ U[ext_new], context ~ U[ext_ctx]); optional padding rows after
    them; the token count is padded to a multiple of ``token_multiple``.
    """
    rng = np.random.default_rng(seed)
    c_dec = rng.integers(dec_ctx[0], dec_ctx[1], size=n_decode, endpoint=True)
    c_ext = rng.integers(ext_ctx[0], ext_ctx[1], size=n_extend, endpoint=True)
    n_ext = rng.integers(ext_new[0], ext_new[1], size=n_extend, endpoint=True)
    ctx = np.concatenate([c_dec, c_ext])
    new = np.concatenate([np.ones(n_decode, np.int64), n_ext])
    T = int(new.sum()) + int(sum(padding_spans or []))
    return build_workload("mixed_step", dtype="bf16", P=4, page_size=16, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, decode=False, ctx_len=ctx, new_len=new,
                          padding_spans=padding_spans,
                          num_tokens=_round_up(max(T, 1), token_multiple), rng=rng, seed=seed)


WORKLOADS = {
    1: tiny_fp32,
    2: gqa_decode,
    3: long_gqa_decode,
    4: mla_decode,
    5: mixed_step,
}


def pool_shape(w: Workload):
    """Physical shape of one pool tensor: [P, num_pages, H_kv, page_size // P, D]."""
    return (w.P, w.num_pages, w.num_kv_heads, w.page_size // w.P, w.head_dim)


def pool_v_shape(w: Workload):
    return (w.P, w.num_pages, w.num_kv_heads, w.page_size // w.P, w.head_dim_v)


def nan_pool(shape, dtype):
    """A pool filled with NaN so that any read of an unwritten slot shows up."""
    return _nan_like(shape, dtype)


def history_tokens(w: Workload):
    """Tokens already in the pool before the step (every real row's context).

    Returns (qo_indptr [B+1], positions [n], k [n, Hkv, D], v [n, Hkv, Dv] or None):
    a "prefill" batch that writes each row's positions 0..ctx-1 through the
    same write entry point the step uses.
    """
    B = w.num_rows
    ctx = np.where(np.arange(B) < w.num_real_rows, w.ctx_len, 0).astype(np.int64)
    qo = np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)
    n = int(qo[-1])
    pos = np.empty((n,), np.int32)
    take = np.empty((n,), np.int64)
    for b in range(B):
        c = int(ctx[b])
        pos[qo[b]: qo[b] + c] = np.arange(c, dtype=np.int32)
        take[qo[b]: qo[b] + c] = w.seq_indptr[b] + np.arange(c)
    k = w.k_seq[take]
    v = None if w.v_seq is None else w.v_seq[take]
    return qo, pos, k, v
