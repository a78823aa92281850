"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Bars: bit-exact pool contents after cp_kv_write; final outputs within max-abs
1e-2 (bf16 output) and LSE within 1e-3 (fp32 workloads: 1e-5 for both);
per-partner fp32 partials within 1e-4 (bf16 inputs) / 1e-5 (fp32 inputs).
Padding tokens must come out exactly 0 / -inf, and NaN planted in padding
rows, padding tokens, the sink page and unwritten pool slots must reach no
real output.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from context_paged_attention_gb300 import workloads as W
from helpers import (OracleView, assert_close, assert_close_lse, assert_within_bound, f64, raw, tolerances,
                     within_bound)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _att(w, **kw):
    from context_paged_attention_gb300.step import StripedAttention

    return StripedAttention(w, device="cuda", **kw)


SMALL = {
    "tiny_fp32": lambda: W.tiny_fp32(),
    "gqa_decode": lambda: W.gqa_decode(seed=21, batch=6, len_lo=20, len_hi=5000),
    "gqa_decode_padded": lambda: W.gqa_decode(seed=22, batch=5, len_lo=1, len_hi=900, padding_spans=[1, 1, 1]),
    "long_gqa_decode": lambda: W.long_gqa_decode(seed=23, batch=2, len_lo=3000, len_hi=20000),
    "mla_decode": lambda: W.mla_decode(seed=24, batch=3, len_lo=100, len_hi=5000),
    "mla_decode_split": lambda: W.mla_decode(seed=30, batch=3, len_lo=9000, len_hi=20000),
    "mla_decode_short": lambda: W.mla_decode(seed=31, batch=4, len_lo=1, len_hi=40),
    # many tokens of 1-4 logical pages: the fused split over clusters charges
    # each token start as 16 pages, so some cluster ranges end inside a
    # token's start cost and hold none of its pages
    "mla_many_short": lambda: W.mla_decode(seed=50, batch=40, len_lo=1, len_hi=200),
    # MLA rows of several new tokens (pool partial + causal own-token partial), padding rows after them
    "mla_mixed": lambda: W.build_workload("mla_mixed", dtype="bf16", P=4, page_size=64, num_q_heads=128,
                                          num_kv_heads=1, head_dim=576, head_dim_v=512, mla=True, decode=False,
                                          scale=1.0 / 192 ** 0.5, ctx_len=[700, 0, 3000, 64, 1500],
                                          new_len=[1, 9, 5, 33, 1], padding_spans=[0, 3], num_tokens=64, seed=40),
    # page 16 with P 4: 4-row page runs, copied with cp.async instead of TMA
    "mla_decode_ps16": lambda: W.build_workload("mla_ps16", dtype="bf16", P=4, page_size=16, num_q_heads=128,
                                                num_kv_heads=1, head_dim=576, head_dim_v=512, mla=True,
                                                scale=1.0 / 192 ** 0.5, ctx_len=[30, 700, 2600],
                                                new_len=[1, 1, 1], seed=32),
    "mixed_step": lambda: W.mixed_step(seed=25, n_decode=4, n_extend=3, dec_ctx=(1, 3000), ext_new=(2, 40),
                                       ext_ctx=(0, 1500), token_multiple=64),
    "mixed_padded": lambda: W.mixed_step(seed=26, n_decode=3, n_extend=3, dec_ctx=(5, 700), ext_new=(2, 17),
                                         ext_ctx=(0, 0), padding_spans=[0, 4, 0, 2], token_multiple=32),
    "gqa_P1": lambda: W.build_workload("gqa_P1", dtype="bf16", P=1, page_size=16, num_q_heads=16,
                                       num_kv_heads=8, head_dim=128, ctx_len=[0, 15, 16, 700, 33],
                                       new_len=[1] * 5, seed=27),
    "gqa_g1_d64": lambda: W.build_workload("gqa_g1_d64", dtype="bf16", P=2, page_size=8, num_q_heads=4,
                                           num_kv_heads=4, head_dim=64, ctx_len=[3, 400, 1], new_len=[1] * 3,
                                           seed=28),
    # interleaved pools: runs of I page offsets per partner (I * P = page size is whole-run pages)
    "tiny_fp32_I4": lambda: W.interleaved(W.tiny_fp32(), 4),
    "gqa_decode_I2": lambda: W.interleaved(W.gqa_decode(seed=33, batch=5, len_lo=1, len_hi=3000), 2),
    "gqa_decode_I4": lambda: W.interleaved(W.gqa_decode(seed=34, batch=5, len_lo=1, len_hi=3000,
                                                        padding_spans=[2, 1]), 4),
    "mla_decode_I16": lambda: W.interleaved(W.mla_decode(seed=35, batch=3, len_lo=1, len_hi=9000), 16),
    "mla_decode_I2": lambda: W.interleaved(W.mla_decode(seed=36, batch=3, len_lo=30, len_hi=3000), 2),
    "mixed_I2": lambda: W.interleaved(W.mixed_step(seed=37, n_decode=3, n_extend=3, dec_ctx=(1, 2000),
                                                   ext_new=(2, 40), ext_ctx=(0, 1500), token_multiple=64), 2),
    # FP8 E4M3 pools with per-tensor descales (decode rows)
    "gqa_decode_fp8": lambda: W.gqa_decode_fp8(seed=38, batch=6, len_lo=20, len_hi=5000),
    "gqa_decode_fp8_I2_pad": lambda: W.interleaved(W.gqa_decode_fp8(seed=39, batch=5, len_lo=1, len_hi=2000,
                                                                    padding_spans=[1, 1]), 2),
    "mixed_fp8": lambda: W.fp8_pool(W.mixed_step(seed=43, n_decode=3, n_extend=3, dec_ctx=(1, 2000), ext_new=(2, 40),
                                                  ext_ctx=(0, 1500), token_multiple=64), 0.0123, 0.0137),
    # stripes longer than the 2048-key split-KV chunk: the chunk merges of the
    # decode kernel, of the multi-token kernel (bulk-copy merge, batches of
    # token rows) and of the E4M3 kernels
    "gqa_decode_split": lambda: W.gqa_decode(seed=44, batch=4, len_lo=8300, len_hi=13000),
    "gqa_decode_fp8_split": lambda: W.gqa_decode_fp8(seed=45, batch=3, len_lo=8300, len_hi=12000),
    "mixed_split": lambda: W.mixed_step(seed=46, n_decode=1, n_extend=2, dec_ctx=(8300, 8600), ext_new=(33, 40),
                                        ext_ctx=(8300, 8700), token_multiple=64),
    "mixed_fp8_split": lambda: W.fp8_pool(W.mixed_step(seed=47, n_decode=1, n_extend=1, dec_ctx=(100, 900),
                                                       ext_new=(33, 36), ext_ctx=(8300, 8600), token_multiple=64),
                                          0.0123, 0.0137),
    "gqa_fp8_g1_d64": lambda: W.fp8_pool(W.build_workload("gqa_fp8_g1_d64", dtype="bf16", P=2, page_size=8,
                                                          num_q_heads=4, num_kv_heads=4, head_dim=64,
                                                          ctx_len=[3, 400, 1], new_len=[1] * 3, seed=40),
                                         0.0091, 0.0213),
    # non-decode steps at other shapes: group 16 / D 64, group 1 / D 128, padded token count
    "mixed_g16_d64": lambda: W.build_workload("mixed_g16_d64", dtype="bf16", P=2, page_size=8, num_q_heads=16,
                                              num_kv_heads=1, head_dim=64, decode=False, ctx_len=[0, 5, 40, 300],
                                              new_len=[3, 1, 17, 70], num_tokens=96, seed=41),
    "mixed_g1": lambda: W.build_workload("mixed_g1", dtype="bf16", P=4, page_size=16, num_q_heads=4,
                                         num_kv_heads=4, head_dim=128, decode=False, ctx_len=[100, 0, 2000],
                                         new_len=[40, 9, 2], seed=42),
    # group 16 (the head-rows decode kernel), one partner with interleave 4; E4M3 at group 16, D 64
    "gqa_g16_P1_I4": lambda: W.interleaved(W.build_workload("gqa_g16_P1", dtype="bf16", P=1, page_size=16,
                                                            num_q_heads=32, num_kv_heads=2, head_dim=128,
                                                            ctx_len=[0, 37, 900], new_len=[1] * 3, seed=44), 4),
    "gqa_fp8_g16_d64": lambda: W.fp8_pool(W.build_workload("gqa_fp8_g16_d64", dtype="bf16", P=2, page_size=8,
                                                           num_q_heads=16, num_kv_heads=1, head_dim=64,
                                                           ctx_len=[5, 300, 1200], new_len=[1] * 3, seed=45),
                                          0.0102, 0.0187),
    "gqa_P16_ps16": lambda: W.build_workload("gqa_P16_ps16", dtype="bf16", P=16, page_size=16, num_q_heads=16,
                                             num_kv_heads=2, head_dim=128, ctx_len=[5, 40, 2000], new_len=[1] * 3,
                                             seed=29),
}


@pytest.fixture(scope="module", params=sorted(SMALL))
def small(request):
    w = SMALL[request.param]()
    att = _att(w)
    att.run_step()
    torch.cuda.synchronize()
    return w, att


def _expected_pool(w, which_v=False):
    """Oracle image: NaN pool, every row's context and the step's new tokens written by the placement."""
    shape = W.pool_v_shape(w) if which_v else W.pool_shape(w)
    fp8 = w.kv_dtype == "fp8"
    if fp8:
        pool = np.full(shape, 0x7F, dtype=np.uint8)  # the E4M3 NaN code
    else:
        dt_nan = W.nan_pool((1,), w.dtype)[0]
        pool = np.full(shape, dt_nan, dtype=np.uint16 if w.dtype == "bf16" else np.float32)
    src = w.v_seq if which_v else w.k_seq
    descale = w.v_descale if which_v else w.k_descale
    for b in range(w.num_real_rows):
        L = int(w.ctx_len[b] + w.new_len[b])
        s0 = int(w.seq_indptr[b])
        rows = w.kv_page_indices[w.kv_page_indptr[b]: w.kv_page_indptr[b + 1]]
        vals = src[s0: s0 + L]
        if fp8:
            vals = oracle.e4m3_quantize(vals, descale)
        pool = oracle.expected_pool_image(pool, rows, np.arange(L), vals, w.page_size, w.P, w.interleave)
    return pool


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def test_kv_write_bit_exact(small):
    w, att = small
    got = raw(att.pool_k)
    want = _expected_pool(w)
    assert np.array_equal(_bits(got), _bits(want)), "pool_k differs from the placement image"
    if not w.mla:
        assert np.array_equal(_bits(raw(att.pool_v)), _bits(_expected_pool(w, True)))
    assert att.status() == 0


def partial_tolerances(w):
    """(O, LSE) bars for one partner's fp32 partial.

    fp32 inputs: 1e-5.  bf16 GQA decode rows: 1e-4 (P V keeps fp32-grade
    probabilities).  MLA and the multi-token rows of non-decode steps: the
    bound of bf16_p_bound, per head and value (None here).  LSEs come from
    fp32 sums: 1e-4.
    """
    if w.dtype == "fp32":
        return 1e-5, 1e-5
    if w.mla or not w.decode:
        return None, 1e-4
    return 1e-4, 1e-4


BF16_P_REL = 2.0 ** -9  # round-to-nearest bf16: relative error of each probability


def bf16_p_bound(A):
    """Bar on a partial whose P V took the probabilities in bf16.

    With weights w_k = p_k / sum p and p~_k = p_k (1 + d_k), |d_k| <= 2^-9:
    normalised by the rounded sum, O~ - O = (sum w_k d_k v_k - dbar O) /
    (1 + dbar) with dbar = sum w_k d_k, so |O~ - O| <= 2^-9 (A + |O|) /
    (1 - 2^-9) <= 2^-8 A / (1 - 2^-9), A = sum w_k |v_k| (per head and value;
    |O| <= A); normalised by the fp32 sum it is <= 2^-9 A.  A 10% allowance
    and 2e-5 absolute cover the fp32 scores, the ex2 approximation and the
    fp32 accumulation, orders of magnitude below at these lengths.
    """
    return 1.1 * 2.0 * BF16_P_REL / (1.0 - BF16_P_REL) * A + 2e-5


def test_partner_partials(small):
    w, att = small
    ov = OracleView(w)
    tol_o, tol_l = partial_tolerances(w)
    o_parts = att.o_parts.cpu().numpy().astype(np.float64)
    l_parts = att.lse_parts.cpu().numpy().astype(np.float64)
    for t in range(w.num_tokens):
        for p in range(w.P):
            if tol_o is None and ov.row_of_token(t) >= 0:
                O, L, A, _ = ov.stripe_abs(t, p)
                assert_within_bound(o_parts[p, t], O, bf16_p_bound(A), f"O part p={p} t={t}")
            else:
                O, L = ov.stripe(t, p)
                assert_close(o_parts[p, t], O, 1e-2 if tol_o is None else tol_o, f"O part p={p} t={t}")
            assert_close_lse(l_parts[p, t], L, tol_l, f"LSE part p={p} t={t}")


@pytest.mark.parametrize("name", ["mla_decode", "mla_decode_I16"])
def test_partial_bar_catches_one_dropped_key(name):
    """The per-head bound is tight enough that an oracle missing one key of
    one partner's stripe (the mistake planted in the oracle, on the host)
    no longer matches the device partial, while the true oracle does."""
    w = SMALL[name]()
    att = _att(w)
    att.run_step()
    torch.cuda.synchronize()
    assert att.status() == 0
    ov = OracleView(w)
    o_parts = att.o_parts.cpu().numpy().astype(np.float64)
    checked = 0
    for t in range(int(w.qo_indptr[w.num_real_rows])):
        p = t % w.P
        O, _, A, n = ov.stripe_abs(t, p)
        if n < 2:
            continue
        bound = bf16_p_bound(A)
        assert within_bound(o_parts[p, t], O, bound), f"t={t} p={p}: the true oracle must match"
        Od, _, _, _ = ov.stripe_abs(t, p, drop=n // 2)  # a key from the middle of the stripe
        assert not within_bound(o_parts[p, t], Od, bound), f"t={t} p={p}: a dropped key went unnoticed"
        checked += 1
        if checked == 4:
            break
    assert checked > 0


def test_step_matches_oracle(small):
    w, att = small
    ov = OracleView(w)
    O, L = ov.final()
    tol_o, tol_l = tolerances(w)
    got_o = f64(att.out)
    got_l = att.lse.cpu().numpy().astype(np.float64)
    assert_close(got_o, O, tol_o, "merged output")
    assert_close_lse(got_l, L, tol_l, "merged LSE")
    # padding tokens merge to exactly 0 / -inf
    t0 = int(w.qo_indptr[w.num_real_rows])
    assert np.all(got_o[t0:] == 0) and np.all(got_l[t0:] == -np.inf)


def test_fused_step_matches_oracle(small):
    """Partials merged inside the partial launch: same bar as partial + lse_merge."""
    w, att = small
    out = torch.empty_like(att.out)
    lse = torch.empty_like(att.lse)
    att.run_step_fused(out=out, lse=lse)
    torch.cuda.synchronize()
    assert att.status() == 0
    O, L = OracleView(w).final()
    tol_o, tol_l = tolerances(w)
    got_o = f64(out)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert_close(got_o, O, tol_o, "fused output")
    assert_close_lse(got_l, L, tol_l, "fused LSE")
    t0 = int(w.qo_indptr[w.num_real_rows])
    assert np.all(got_o[t0:] == 0) and np.all(got_l[t0:] == -np.inf)
    # and against the two-launch path on the device: both are within tol_o of
    # the oracle, and they sum in different orders (the fused MLA kernel over
    # pages merges the partners inside its softmax), so two independent
    # round-to-nearest bf16 outputs may sit one unit apart (2^-6 near 2.5):
    # within 2 tol_o of each other
    assert_close(got_o, f64(att.out), 2 * tol_o, "fused vs partial + merge")


def test_head_major_lse_partial(small):
    """cp_paged_attn_partial_ex with [P][H][T] LSEs writes the same values."""
    w, att = small
    from context_paged_attention_gb300 import binding as B
    P, T, Hq = w.P, w.num_tokens, w.num_q_heads
    o = torch.empty_like(att.o_parts[:P])
    l_hm = torch.empty((P, Hq, T), dtype=torch.float32, device=att.device)
    one_per_row = w.decode and w.num_tokens == w.num_rows
    B.cp_paged_attn_partial_ex(att.desc, att.pool_k, att.pool_v, att.q, att.kv_len, att.max_kv_len, att.page_indptr,
                               att.page_indices, w.scale, o, l_hm, att.workspace, lse_layout=B.LSE_HEAD_MAJOR,
                               qo_indptr=None if one_per_row else att.qo_indptr, num_rows=w.num_rows,
                               dev_status=att.dev_status)
    torch.cuda.synchronize()
    assert att.status() == 0
    assert torch.equal(o, att.o_parts[:P])
    assert torch.equal(l_hm.transpose(1, 2), att.lse_parts[:P])


def test_plain_partial_entry(small):
    """cp_paged_attn_partial (natural row order, token-major LSE) writes the
    same partials as the step's cp_paged_attn_partial_ex (longest rows first)."""
    w, att = small
    from context_paged_attention_gb300 import binding as B
    P = w.P
    o = torch.empty_like(att.o_parts[:P])
    lse = torch.empty_like(att.lse_parts[:P])
    one_per_row = w.decode and w.num_tokens == w.num_rows
    B.cp_paged_attn_partial(att.desc, att.pool_k, att.pool_v, att.q, att.kv_len, att.max_kv_len, att.page_indptr,
                            att.page_indices, w.scale, o, lse, att.workspace,
                            qo_indptr=None if one_per_row else att.qo_indptr, num_rows=w.num_rows,
                            dev_status=att.dev_status)
    torch.cuda.synchronize()
    assert att.status() == 0
    assert torch.equal(o, att.o_parts[:P]) and torch.equal(lse, att.lse_parts[:P])


def test_tp_mode_step(small):
    """TP-mode head layout: per-rank combine of head slices from head-major
    LSEs, then the own-token merge, equals the plain attention."""
    w, att = small
    if w.num_q_heads % w.P != 0:
        pytest.skip("query heads do not split over the P ranks")
    out = torch.empty_like(att.out)
    lse = torch.empty_like(att.lse)
    att.run_step_tp(out=out, lse=lse)
    torch.cuda.synchronize()
    assert att.status() == 0
    O, L = OracleView(w).final()
    tol_o, tol_l = tolerances(w)
    got_o = f64(out)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert_close(got_o, O, tol_o, "TP-mode output")
    assert_close_lse(got_l, L, tol_l, "TP-mode LSE")
    t0 = int(w.qo_indptr[w.num_real_rows])
    assert np.all(got_o[t0:] == 0) and np.all(got_l[t0:] == -np.inf)


def test_own_token_partial(small):
    w, att = small
    if w.decode:
        pytest.skip("decode steps attend the pool only")
    ov = OracleView(w)
    o_own = att.o_parts[w.P].cpu().numpy().astype(np.float64)
    l_own = att.lse_parts[w.P].cpu().numpy().astype(np.float64)
    for b in range(w.num_real_rows):
        s0 = int(w.seq_indptr[b])
        c, n = int(w.ctx_len[b]), int(w.new_len[b])
        K = oracle.raw_to_f64(w.k_seq[s0 + c: s0 + c + n])
        if w.mla:
            K, V = oracle.mla_kv(K, w.head_dim_v)
        else:
            V = oracle.raw_to_f64(w.v_seq[s0 + c: s0 + c + n])
        t0 = int(w.qo_indptr[b])
        O, L = oracle.causal_own_attention(ov.q[t0: t0 + n], K, V, w.scale)
        assert_close(o_own[t0: t0 + n], O, 1e-4, f"own O row {b}")
        assert_close_lse(l_own[t0: t0 + n], L, 1e-4, f"own LSE row {b}")
    t0 = int(w.qo_indptr[w.num_real_rows])
    assert np.all(o_own[t0:] == 0) and np.all(l_own[t0:] == -np.inf)


def test_repeat_step_is_stable(small):
    """Running the step again (same write, same tables) gives bit-identical outputs."""
    w, att = small
    first = raw(att.out).copy()
    att.run_step()
    torch.cuda.synchronize()
    assert np.array_equal(_bits(raw(att.out)), _bits(first))


# ---------------------------------------------------------------- full-size workloads

FULL = {
    "gqa_decode": (W.gqa_decode, None),
    "gqa_decode_fp8": (W.gqa_decode_fp8, [0, 9, 63]),
    "long_gqa_decode": (W.long_gqa_decode, list(range(8))),
    "mla_decode": (W.mla_decode, [0, 4, 7, 12, 19, 23, 27, 31]),
    "mixed_step": (W.mixed_step, [0, 17, 47, 48, 55, 63]),
}


@pytest.mark.parametrize("n", [1, 5, 32, 33, 40])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_lse_merge_partial_counts(n, out_bf16):
    """Contiguous-partial merge against the oracle merge for partial counts on
    both sides of the warp width (weights held one a lane up to 32), with
    empty partials and a token whose partials are all empty."""
    from context_paged_attention_gb300 import binding as B
    rng = np.random.default_rng(100 + n)
    T, H, Dv = 29, 3, 128
    O = rng.standard_normal((n, T, H, Dv))
    L = rng.standard_normal((n, T, H)) * 3
    L[rng.random((n, T, H)) < 0.25] = -np.inf
    L[:, 4, :] = -np.inf
    dev = torch.device("cuda")
    o_d = torch.tensor(O, dtype=torch.float32, device=dev)
    l_d = torch.tensor(L, dtype=torch.float32, device=dev)
    out = torch.zeros((T, H, Dv), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
    lse = torch.zeros((T, H), dtype=torch.float32, device=dev)
    B.lse_merge(o_d, l_d, out, lse)
    torch.cuda.synchronize()
    O32 = o_d.cpu().numpy().astype(np.float64)
    L32 = l_d.cpu().numpy().astype(np.float64)
    want_o = np.zeros((T, H, Dv))
    want_l = np.zeros((T, H))
    for t in range(T):
        want_o[t], want_l[t] = oracle.merge(O32[:, t], L32[:, t])
    got_o = out.float().cpu().numpy().astype(np.float64)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert np.all(got_o[4] == 0.0) and np.all(np.isneginf(got_l[4]))
    assert_close(got_o, want_o, 1e-2 if out_bf16 else 1e-5, "merged O")
    fin = np.isfinite(want_l)
    assert np.array_equal(fin, np.isfinite(got_l))
    assert_close(got_l[fin], want_l[fin], 1e-5, "merged LSE")


@pytest.mark.parametrize("n,layout", [(1, "th"), (3, "ht"), (5, "mixed"), (16, "mixed")])
def test_lse_merge_views(n, layout):
    """Strided-view merge against the oracle merge on random partials (some
    empty), LSEs token- or head-major, output into a head slice."""
    from context_paged_attention_gb300 import binding as B
    rng = np.random.default_rng(n)
    T, H, Dv = 37, 6, 64
    O = rng.standard_normal((n, T, H, Dv))
    L = rng.standard_normal((n, T, H)) * 3
    L[rng.random((n, T, H)) < 0.2] = -np.inf
    L[:, 5, :] = -np.inf  # a token with every partial empty
    dev = torch.device("cuda")
    o_d = torch.tensor(O, dtype=torch.float32, device=dev)
    views, keep = [], []
    for i in range(n):
        hm = layout == "ht" or (layout == "mixed" and i % 2 == 1)
        lt = torch.tensor(L[i].T.copy() if hm else L[i], dtype=torch.float32, device=dev)
        keep.append(lt)
        views.append(B.view(o_d, lt, H * Dv, Dv, 1 if hm else H, T if hm else 1, o_offset=i * T * H * Dv))
    Hout = H + 2  # write heads 1 .. H of a wider output
    out = torch.zeros((T, Hout, Dv), dtype=torch.float32, device=dev)
    lse = torch.zeros((Hout, T), dtype=torch.float32, device=dev)  # head-major LSE out
    B.lse_merge_views(views, T, H, Dv, out, Hout * Dv, Dv, lse, 1, T, out_offset=Dv, lse_out_offset=T)
    torch.cuda.synchronize()
    O32 = o_d.cpu().numpy().astype(np.float64)
    L32 = np.asarray(L, dtype=np.float32).astype(np.float64)
    want_o = np.zeros((T, H, Dv))
    want_l = np.zeros((T, H))
    for t in range(T):
        want_o[t], want_l[t] = oracle.merge(O32[:, t], L32[:, t])
    got_o = out.cpu().numpy().astype(np.float64)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert_close(got_o[:, 1:H + 1], want_o, 1e-5, "merged view output")
    assert_close_lse(got_l[1:H + 1].T, want_l, 1e-5, "merged view LSE")
    assert np.all(got_o[:, 0] == 0) and np.all(got_o[:, H + 1] == 0) and np.all(got_l[0] == 0)


@pytest.mark.parametrize("name,fused", [("gqa_decode", True), ("mixed_step", True), ("mla_decode", True),
                                        ("gqa_decode", False), ("mixed_step", False)])
def test_graph_replay(name, fused):
    """A step captured as a CUDA graph (fused, or partial + merge): replays
    equal the eager call bit for bit, and a replay after refilling the inputs
    gives the new step."""
    w = SMALL[name]()
    att = _att(w)
    out0, lse0 = att.run_step_fused() if fused else att.run_step()
    ref_o, ref_l = out0.clone(), lse0.clone()
    att.capture(fused)
    for _ in range(2):
        o, l_ = att.replay()
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16) if o.dtype == torch.bfloat16 else o,
                           ref_o.view(torch.int16) if ref_o.dtype == torch.bfloat16 else ref_o)
        assert torch.equal(l_, ref_l)
    # new step values in the captured buffers: queries doubled (exact in bf16)
    att.q.mul_(2)
    o, l_ = att.replay()
    torch.cuda.synchronize()
    assert att.status() == 0
    q2 = W.f32_to_bf16_bits(2 * oracle.raw_to_f64(w.q).astype(np.float32)) if w.dtype == "bf16" else 2 * w.q
    w2 = dataclasses.replace(w, q=q2)
    O, L = OracleView(w2).final()
    tol_o, tol_l = tolerances(w)
    assert_close(f64(o), O, tol_o, "replayed output")
    assert_close_lse(l_.cpu().numpy().astype(np.float64), L, tol_l, "replayed LSE")


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_size_sampled(name):
    fn, rows = FULL[name]
    w = fn()
    att = _att(w)
    att.run_step()
    torch.cuda.synchronize()
    assert att.status() == 0
    got_o = f64(att.out)
    got_l = att.lse.cpu().numpy().astype(np.float64)
    # properties over every output: finite for real tokens, exact 0 / -inf for padding
    t_end = int(w.qo_indptr[w.num_real_rows])
    assert np.all(np.isfinite(got_o[:t_end])) and np.all(np.isfinite(got_l[:t_end]))
    assert np.all(got_o[t_end:] == 0) and np.all(got_l[t_end:] == -np.inf)
    assert np.all(np.abs(got_o[:t_end]) <= 7.0)  # convex combination of N(0,1) draws
    ov = OracleView(w)
    tol_o, tol_l = tolerances(w)
    row_list = range(w.num_real_rows) if rows is None else rows
    rng = np.random.default_rng(7)
    # every head of the sampled rows for the MLA and long-context workloads (8 rows each)
    all_heads = name in ("mla_decode", "long_gqa_decode")
    for b in row_list:
        heads = None if (rows is None or all_heads) else sorted(
            rng.choice(w.num_q_heads, size=8, replace=False).tolist())
        O, L = ov.final_row(b, heads)
        t0, n = int(w.qo_indptr[b]), int(w.new_len[b])
        sel_o = got_o[t0: t0 + n] if heads is None else got_o[t0: t0 + n][:, heads]
        sel_l = got_l[t0: t0 + n] if heads is None else got_l[t0: t0 + n][:, heads]
        assert_close(sel_o, O, tol_o, f"{name} row {b} O")
        assert_close_lse(sel_l, L, tol_l, f"{name} row {b} LSE")


# ---------------------------------------------------------------- device-side checks

def test_bad_page_id_is_reported_not_read():
    """A page id outside the pool is skipped and reported; other rows are unaffected."""
    w = W.gqa_decode(seed=31, batch=4, len_lo=100, len_hi=400)
    att = _att(w)
    att.run_step()
    torch.cuda.synchronize()
    good = raw(att.out).copy()
    b = 2
    idx = att.page_indices.clone()
    idx[int(w.kv_page_indptr[b])] = w.num_pages + 1000  # far outside the pool
    att.page_indices = idx
    att.partial()
    att.merge()
    torch.cuda.synchronize()
    assert att.status() == 1  # CPATTN_DEV_PAGE_OUT_OF_RANGE
    out = raw(att.out)
    for r in range(w.num_rows):
        if r != b:
            assert np.array_equal(_bits(out[r]), _bits(good[r]))


def test_kv_len_past_table_is_reported():
    w = W.gqa_decode(seed=32, batch=3, len_lo=50, len_hi=90)
    att = _att(w)
    att.run_step()
    torch.cuda.synchronize()
    kv = att.kv_len.clone()
    kv[1] = int(w.kv_len[1]) + 10 * w.page_size  # beyond the row's page table
    att.kv_len = kv
    att.max_kv_len = int(kv.max().item())
    from context_paged_attention_gb300 import binding as B

    ws = B.workspace_bytes(att.desc, w.num_q_heads, w.num_tokens, att.max_kv_len)
    att.workspace = torch.empty((max(ws, 256),), dtype=torch.uint8, device="cuda")
    att.partial()
    torch.cuda.synchronize()
    assert att.status() == 2  # CPATTN_DEV_POS_PAST_TABLE
