"""float64 reference for striped (context-parallel) paged attention.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Straightforward NumPy,
one head at a time, no blocking, fusion or reordering beyond the definitions.

Readings taken where the pages leave a step open (each is listed with its
reason in the design notes of the repository):

* The striping index ``s`` is the slot offset inside a logical page.  With the
  page size a multiple of P this gives the same partner and physical slot as
  using the global slot number, and a partner page holds ``page_size // P``
  slots.
* An interleave size I (named by the vLLM page, cp_kv_cache_interleave_size,
  without a formula) moves runs of I consecutive offsets together: partner
  ``(off // I) % P``, physical slot ``(off // (I * P)) * I + off % I``.
* The log-sum-exp is the natural logarithm.
* Grouped-query heads: query head ``h`` reads KV head ``h // (Hq // Hkv)``.
* A decode row attends every key of its row, its own (just written) key
  included; a row of a non-decode step has a context of ``c`` keys in the pool
  and its ``i``-th new token (0-based) additionally sees new tokens ``0..i``.
* MLA: one latent row of ``D_qk`` values per token serves as the key; its
  first ``D_v`` values are the value.
* An empty key set gives output 0 and log-sum-exp -inf; merging only such
  partials gives 0 and -inf again (padding merges to zero).
* FP8 pools (the vLLM page passes per-tensor ``k_descale`` / ``v_descale`` to
  the attention call): keys and values are stored as OCP FP8 E4M3 codes of
  ``x / descale`` (quotient in float32, rounded to the nearest E4M3 value,
  ties to even, magnitudes past 448 saturated to 448) and read back as
  ``code value * descale``; queries stay in their own type.
"""

from __future__ import annotations

import bisect

import numpy as np

NEG_INF = -np.inf


# --------------------------------------------------------------------------
# value conversion (raw input arrays -> exact float64)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """Value of an FP8 E4M3 code (OCP 8-bit floating point, E4M3 variant):
    sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 holds
    the subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table() -> np.ndarray:
    """float64 values of all 256 codes (NaN for the two NaN codes)."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(x: float, _vals=None) -> int:
    """Nearest E4M3 code to x: ties go to the even code, magnitudes beyond
    448 saturate to 448, NaN gives 0x7F.  Written as a search over the 127
    non-negative finite codes, whose values increase with the code
    (``_vals``: their values, when the caller already has them)."""
    x = float(x)
    if x != x:
        return 0x7F
    neg = np.signbit(x)
    a = min(abs(x), E4M3_MAX)
    vals = _vals if _vals is not None else [e4m3_value(c) for c in range(0x7F)]  # codes 0x00 .. 0x7E
    lo = bisect.bisect_right(vals, a) - 1  # largest code whose value is <= a
    if vals[lo] == a or lo == 0x7E:
        code = lo
    else:
        hi = lo + 1
        d_lo, d_hi = a - vals[lo], vals[hi] - a
        code = lo if d_lo < d_hi else hi if d_hi < d_lo else (lo if lo % 2 == 0 else hi)
    return code | (0x80 if neg else 0)


def e4m3_quantize(x_raw: np.ndarray, descale: float) -> np.ndarray:
    """Codes stored for raw values (bf16 bits or float32) with a per-tensor
    descale: E4M3 code of float32(x) / float32(descale), the quotient rounded
    to float32 first."""
    x = raw_to_f64(x_raw).astype(np.float32)
    qt = (x / np.float32(descale)).astype(np.float32)
    vals = [e4m3_value(c) for c in range(0x7F)]
    # each distinct quotient is encoded once (bf16 inputs have few distinct
    # values); distinct by bit pattern, so -0.0 keeps its sign (code 0x80)
    uniq, inv = np.unique(qt.reshape(-1).view(np.uint32), return_inverse=True)
    codes = np.array([e4m3_encode(float(v), vals) for v in uniq.view(np.float32)], dtype=np.uint8)
    return codes[inv].reshape(qt.shape)


def e4m3_dequantize(codes: np.ndarray, descale: float) -> np.ndarray:
    """float64 values of stored codes: code value * descale."""
    return e4m3_table()[np.asarray(codes, dtype=np.uint8)] * float(descale)

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 numbers given as uint16 bit patterns.

    A bfloat16 is the upper half of an IEEE float32, so the value is the
    float32 whose high 16 bits are ``bits`` and whose low 16 bits are zero.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def raw_to_f64(raw: np.ndarray) -> np.ndarray:
    """float64 view of an input array: uint16 means bfloat16 bits, float32 is itself."""
    raw = np.asarray(raw)
    if raw.dtype == np.uint16:
        return bf16_bits_to_f64(raw)
    if raw.dtype == np.float32 or raw.dtype == np.float64:
        return raw.astype(np.float64)
    raise TypeError(f"unsupported raw dtype {raw.dtype}")


# --------------------------------------------------------------------------
# placement (mstar PR #1124, description: striped context-parallel pool)
# --------------------------------------------------------------------------

def placement(page_row, pos: int, page_size: int, P: int, interleave: int = 1):
    """Where logical position ``pos`` of a row lives in a P-way striped pool.

    The row's page table ``page_row`` lists logical page ids.  The token sits
    in logical page ``page_row[pos // page_size]`` at offset
    ``off = pos % page_size``.  The pool stripes each page's slots over the P
    partners: offset ``off`` belongs to partner ``off % P`` and is that
    partner's physical slot ``off // P`` inside the *same* page id (page ids
    stay logical).  Returns ``(partner, page_id, physical_slot)``.

    With an interleave size I > 1 (vLLM's cp_kv_cache_interleave_size), runs
    of I consecutive offsets go to one partner: offset ``off`` belongs to
    partner ``(off // I) % P`` at physical slot ``(off // (I * P)) * I + off % I``
    (I = 1 is the striping above).  I * P must divide the page size.
    """
    if P <= 0 or interleave <= 0 or page_size % (P * interleave) != 0:
        raise ValueError("P * interleave must divide page_size")
    page = int(page_row[pos // page_size])
    off = pos % page_size
    grp = off // interleave
    return grp % P, page, (grp // P) * interleave + off % interleave


def placement_inverse(page_row, page: int, phys: int, partner: int, page_size: int, P: int,
                      interleave: int = 1) -> int:
    """Logical position stored at (partner, page id, physical slot); -1 if the
    page is not in the row's table.  Offset in the page is
    ``((phys // I) * P + partner) * I + phys % I`` (``phys * P + partner`` for I = 1)."""
    hits = np.nonzero(np.asarray(page_row) == page)[0]
    if hits.size == 0:
        return -1
    off = ((phys // interleave) * P + partner) * interleave + phys % interleave
    return int(hits[0]) * page_size + off


def stripe_positions(length: int, P: int, p: int, interleave: int = 1) -> np.ndarray:
    """Logical positions of a row of ``length`` keys that partner ``p`` holds,
    in the order of the partner's physical slots.

    Since ``page_size`` is a multiple of P * I, the partner of an offset is
    the partner of the position: ``(pos // I) % P``.
    """
    pos = np.arange(length, dtype=np.int64)
    return pos[(pos // interleave) % P == p]


def expected_pool_image(pool_raw: np.ndarray, page_row, positions, new_raw: np.ndarray,
                        page_size: int, P: int, interleave: int = 1) -> np.ndarray:
    """Pool contents after writing new tokens through the placement.

    ``pool_raw`` has the library's physical layout
    ``[P, num_pages, H_kv, page_size // P, D]``; it is copied, and token ``t``
    (logical position ``positions[t]``, values ``new_raw[t]`` of shape
    ``[H_kv, D]``) is written at ``[partner, page, :, slot, :]``.  Negative
    positions are padding tokens and are not written.
    """
    out = np.array(pool_raw, copy=True)
    for t, pos in enumerate(positions):
        if pos < 0:
            continue
        p, page, slot = placement(page_row, int(pos), page_size, P, interleave)
        out[p, page, :, slot, :] = new_raw[t]
    return out


# --------------------------------------------------------------------------
# attention (plain softmax definition over the logical key sequence)
# --------------------------------------------------------------------------

def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Softmax attention of one query token over ``m`` keys, with its LSE.

    q: [Hq, Dqk], K: [m, Hkv, Dqk], V: [m, Hkv, Dv] (float64).
    For query head h with KV head kh = h // (Hq // Hkv):
        s_j   = scale * <q[h], K[j, kh]>
        LSE   = ln sum_j exp(s_j)       (computed as max + ln sum exp(s - max))
        O[h]  = sum_j exp(s_j - LSE) V[j, kh]
    With m == 0: O = 0 and LSE = -inf.
    Returns (O [Hq, Dv], LSE [Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Hq = q.shape[0]
    m, Hkv = K.shape[0], K.shape[1]
    Dv = V.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("query heads must be a multiple of KV heads")
    g = Hq // Hkv
    O = np.zeros((Hq, Dv), dtype=np.float64)
    LSE = np.full((Hq,), NEG_INF, dtype=np.float64)
    if m == 0:
        return O, LSE
    for h in range(Hq):
        kh = h // g
        s = scale * (K[:, kh, :] @ q[h])
        mx = s.max()
        w = np.exp(s - mx)
        z = w.sum()
        O[h] = (w @ V[:, kh, :]) / z
        LSE[h] = mx + np.log(z)
    return O, LSE


def stripe_partial(q, K, V, scale: float, P: int, p: int, interleave: int = 1):
    """Partner p's partial: attention restricted to the keys partner p holds
    (j % P == p; with interleave I, (j // I) % P == p)."""
    idx = stripe_positions(K.shape[0], P, p, interleave)
    return attention(q, K[idx], V[idx], scale)


def merge(O_parts, LSE_parts):
    """Exact merge of partials over disjoint key sets.

    With M = max_i LSE_i: if M = -inf every partial is empty and the result is
    O = 0, LSE = -inf.  Otherwise w_i = exp(LSE_i - M), LSE = M + ln sum_i w_i
    and O = sum_i w_i O_i / sum_i w_i.  Works per head.
    O_parts: [N, H, Dv], LSE_parts: [N, H].
    """
    O_parts = np.asarray(O_parts, dtype=np.float64)
    LSE_parts = np.asarray(LSE_parts, dtype=np.float64)
    N, H, Dv = O_parts.shape
    O = np.zeros((H, Dv), dtype=np.float64)
    LSE = np.full((H,), NEG_INF, dtype=np.float64)
    for h in range(H):
        mx = LSE_parts[:, h].max()
        if mx == NEG_INF:
            continue
        w = np.exp(LSE_parts[:, h] - mx)
        z = w.sum()
        O[h] = (w @ O_parts[:, h, :]) / z
        LSE[h] = mx + np.log(z)
    return O, LSE


def causal_own_attention(q_new, k_new, v_new, scale: float):
    """Own-token partial of one row of a non-decode step.

    New token i attends the row's new keys 0..i (the K/V the layer passes,
    causal on equal-length query and key spans).
    q_new: [n, Hq, Dqk], k_new: [n, Hkv, Dqk], v_new: [n, Hkv, Dv].
    Returns (O [n, Hq, Dv], LSE [n, Hq]).
    """
    n = q_new.shape[0]
    Hq, Dv = q_new.shape[1], v_new.shape[2]
    O = np.zeros((n, Hq, Dv), dtype=np.float64)
    LSE = np.full((n, Hq), NEG_INF, dtype=np.float64)
    for i in range(n):
        O[i], LSE[i] = attention(q_new[i], k_new[: i + 1], v_new[: i + 1], scale)
    return O, LSE


def mla_kv(latent: np.ndarray, dv: int):
    """MLA reading: the latent row [m, 1, Dqk] is the key, its first dv values the value."""
    return latent, latent[:, :, :dv]


# --------------------------------------------------------------------------
# whole step: the plain definition the striped method must reproduce
# --------------------------------------------------------------------------

def expected_step(q, k_seq, v_seq, seq_indptr, ctx_len, new_len, qo_indptr,
                  num_real_rows: int, num_tokens: int, scale: float,
                  rows=None, heads=None):
    """Final merged output of a step, by the plain definition (no striping).

    For real row b with ``ctx_len[b]`` keys already in the pool and
    ``new_len[b]`` new tokens (query tokens ``qo_indptr[b]..qo_indptr[b+1]``),
    new token i attends the row's logical keys ``0 .. ctx_len[b] + i``.
    For a decode row (ctx = L - 1, one new token) that is all L keys.

    q: [T, Hq, Dqk]; k_seq: [sum L, Hkv, Dqk]; v_seq: [sum L, Hkv, Dv] (float64),
    row b's logical sequence at ``seq_indptr[b]:seq_indptr[b+1]``.
    Tokens of padding rows and tokens past the last real row get O = 0,
    LSE = -inf.  ``rows``/``heads`` restrict the work to a sample (other
    entries stay 0 / -inf).
    Returns (O [T, Hq, Dv], LSE [T, Hq]).
    """
    Hq = q.shape[1]
    Dv = v_seq.shape[2]
    O = np.zeros((num_tokens, Hq, Dv), dtype=np.float64)
    LSE = np.full((num_tokens, Hq), NEG_INF, dtype=np.float64)
    row_list = range(num_real_rows) if rows is None else rows
    for b in row_list:
        base = int(seq_indptr[b])
        for i in range(int(new_len[b])):
            t = int(qo_indptr[b]) + i
            m = int(ctx_len[b]) + i + 1
            Kb = k_seq[base: base + m]
            Vb = v_seq[base: base + m]
            if heads is None:
                O[t], LSE[t] = attention(q[t], Kb, Vb, scale)
            else:
                g = Hq // Kb.shape[1]
                for h in heads:
                    kh = h // g
                    o1, l1 = attention(q[t, h: h + 1], Kb[:, kh: kh + 1], Vb[:, kh: kh + 1], scale)
                    O[t, h], LSE[t, h] = o1[0], l1[0]
    return O, LSE
