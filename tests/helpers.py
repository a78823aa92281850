"""Test helpers: device tensors -> NumPy, oracle views of a workload."""

import numpy as np
import torch

import oracle


def raw(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> host array of its raw values (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return oracle.raw_to_f64(raw(t))


class OracleView:
    """float64 view of a workload's values for the oracle (per-row slices on demand)."""

    def __init__(self, w):
        self.w = w
        self.q = oracle.raw_to_f64(w.q)

    def row_kv(self, b, m):
        w = self.w
        s0 = int(w.seq_indptr[b])
        if w.kv_dtype == "fp8":  # the pool holds E4M3 codes: read back code * descale
            K = oracle.e4m3_dequantize(oracle.e4m3_quantize(w.k_seq[s0: s0 + m], w.k_descale), w.k_descale)
            V = oracle.e4m3_dequantize(oracle.e4m3_quantize(w.v_seq[s0: s0 + m], w.v_descale), w.v_descale)
            return K, V
        K = oracle.raw_to_f64(w.k_seq[s0: s0 + m])
        if w.mla:
            return oracle.mla_kv(K, w.head_dim_v)
        return K, oracle.raw_to_f64(w.v_seq[s0: s0 + m])

    def row_of_token(self, t):
        w = self.w
        for b in range(w.num_real_rows):
            if w.qo_indptr[b] <= t < w.qo_indptr[b + 1]:
                return b
        return -1

    def stripe(self, t, p, heads=None):
        """Oracle partial of partner p for token t (keys the pool partial sees)."""
        w = self.w
        b = self.row_of_token(t)
        Hq = w.num_q_heads
        if b < 0:
            return np.zeros((Hq, w.head_dim_v)), np.full((Hq,), -np.inf)
        m = int(w.kv_len[b])
        K, V = self.row_kv(b, m)
        q = self.q[t] if heads is None else self.q[t][heads]
        if heads is not None:
            g = Hq // w.num_kv_heads
            kh = np.asarray(heads) // g
            # attention per selected head with its own KV head
            O = np.zeros((len(heads), w.head_dim_v))
            L = np.zeros((len(heads),))
            for i, h in enumerate(heads):
                o, l_ = oracle.stripe_partial(q[i: i + 1], K[:, kh[i]: kh[i] + 1], V[:, kh[i]: kh[i] + 1],
                                              w.scale, w.P, p, w.interleave)
                O[i], L[i] = o[0], l_[0]
            return O, L
        return oracle.stripe_partial(q, K, V, w.scale, w.P, p, w.interleave)

    def stripe_abs(self, t, p, drop=None):
        """Partner p's softmax weights applied to |V| (sum_k w_k |v_k| per head
        and value), and the partial itself, for token t; `drop`: index (within
        the stripe) of one key to leave out."""
        w = self.w
        b = self.row_of_token(t)
        m = int(w.kv_len[b])
        K, V = self.row_kv(b, m)
        idx = oracle.stripe_positions(m, w.P, p, w.interleave)
        if drop is not None:
            idx = np.delete(idx, drop)
        q = self.q[t]
        g = w.num_q_heads // w.num_kv_heads
        Hq = w.num_q_heads
        O = np.zeros((Hq, w.head_dim_v))
        A = np.zeros((Hq, w.head_dim_v))
        L = np.zeros((Hq,))
        for kh in range(w.num_kv_heads):
            hs = slice(kh * g, (kh + 1) * g)
            Kk, Vk = K[idx, kh: kh + 1], V[idx, kh: kh + 1]
            O[hs], L[hs] = oracle.attention(q[hs], Kk, Vk, w.scale)
            A[hs], _ = oracle.attention(q[hs], Kk, np.abs(Vk), w.scale)
        return O, L, A, len(idx)

    def final(self, rows=None, heads=None):
        w = self.w
        if w.kv_dtype == "fp8":
            # keys and values as the pool returns them; a non-decode step's own
            # tokens are attended from the step's bf16 K / V, not the pool
            k = oracle.e4m3_dequantize(oracle.e4m3_quantize(w.k_seq, w.k_descale), w.k_descale)
            v = oracle.e4m3_dequantize(oracle.e4m3_quantize(w.v_seq, w.v_descale), w.v_descale)
            if not w.decode:
                for b in range(w.num_real_rows):
                    s0, c, n = int(w.seq_indptr[b]), int(w.ctx_len[b]), int(w.new_len[b])
                    k[s0 + c: s0 + c + n] = oracle.raw_to_f64(w.k_seq[s0 + c: s0 + c + n])
                    v[s0 + c: s0 + c + n] = oracle.raw_to_f64(w.v_seq[s0 + c: s0 + c + n])
        else:
            k = oracle.raw_to_f64(w.k_seq)
            v = oracle.mla_kv(k, w.head_dim_v)[1] if w.mla else oracle.raw_to_f64(w.v_seq)
        return oracle.expected_step(self.q, k, v, w.seq_indptr, w.ctx_len, w.new_len, w.qo_indptr,
                                    w.num_real_rows, w.num_tokens, w.scale, rows=rows, heads=heads)

    def final_row(self, b, heads=None):
        """Oracle output for the tokens of row b only (large workloads)."""
        w = self.w
        n = int(w.new_len[b])
        m = int(w.ctx_len[b]) + n
        K, V = self.row_kv(b, m)
        Hq = w.num_q_heads
        hs = list(range(Hq)) if heads is None else list(heads)
        g = Hq // w.num_kv_heads
        O = np.zeros((n, len(hs), w.head_dim_v))
        L = np.zeros((n, len(hs)))
        for i in range(n):
            t = int(w.qo_indptr[b]) + i
            mm = int(w.ctx_len[b]) + i + 1
            for j, h in enumerate(hs):
                kh = h // g
                o, l_ = oracle.attention(self.q[t, h: h + 1], K[:mm, kh: kh + 1], V[:mm, kh: kh + 1], w.scale)
                O[i, j], L[i, j] = o[0], l_[0]
        return O, L


def tolerances(w):
    """Final-output tolerances: fp32 workloads 1e-5 / 1e-5; bf16 output 1e-2, fp32 LSE 1e-3."""
    return (1e-5, 1e-5) if w.dtype == "fp32" else (1e-2, 1e-3)


def assert_close_lse(got, want, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: -inf pattern differs"
    assert np.all(got[~fin] == -np.inf), f"{what}: empty sets must give -inf"
    if fin.any():
        err = np.max(np.abs(got[fin] - want[fin]))
        assert err <= tol, f"{what}: max |dLSE| {err:.3e} > {tol}"


def within_bound(got, want, bound):
    """Whether |got - want| <= bound elementwise (bound broadcast to the arrays)."""
    d = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    return bool(np.all(np.isfinite(d)) and np.all(d <= bound))


def assert_within_bound(got, want, bound, what=""):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    ratio = float(np.max(d / bound)) if np.size(d) else 0.0
    assert np.all(np.isfinite(d)) and ratio <= 1.0, f"{what}: max |d| / bound {ratio:.3f} > 1"
    return ratio


def assert_close(got, want, tol, what=""):
    err = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64)))) if np.size(want) else 0.0
    assert np.isfinite(err) and err <= tol, f"{what}: max |d| {err:.3e} > {tol}"
    return err
