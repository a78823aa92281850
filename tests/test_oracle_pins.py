"""Pins for the float64 oracle: checks against things other than itself.

Each pin is independent of the oracle code it checks: hand-derived golden
tables (tests/golden), brute force with explicit loops, closed forms, a
library routine (torch scaled_dot_product_attention in float64, scipy
logsumexp), and invariants the pages state (P partners attend like one;
padding merges to zero).  ``test_planted_mistakes_are_caught`` plants
plausible mistakes in the oracle and checks that some pin fails.
"""

import math
import os

import numpy as np
import pytest

import oracle
from oracle import reference as R
from context_paged_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


# ---------------------------------------------------------------- placement

def pin_placement_golden():
    page_row = [5, 2, 7]
    for pos, p, page, slot in _rows("placement_ps8_P4.txt"):
        got = oracle.placement(page_row, int(pos), 8, 4)
        assert got == (int(p), int(page), int(slot)), (pos, got)


def pin_placement_golden_interleaved():
    page_row = [3, 6]
    for pos, p, page, slot in _rows("placement_ps8_P2_I2.txt"):
        got = oracle.placement(page_row, int(pos), 8, 2, 2)
        assert got == (int(p), int(page), int(slot)), (pos, got)


def pin_placement_bijection_interleaved(seed=10):
    """Bijection and inverse with interleave sizes; I = 1 reproduces the striping."""
    rng = np.random.default_rng(seed)
    for ps, P, I in [(16, 2, 2), (16, 4, 4), (64, 4, 2), (64, 8, 8), (32, 1, 4)]:
        pages = rng.permutation(30)[:4]
        seen = set()
        for pos in range(ps * len(pages)):
            p, page, slot = oracle.placement(pages, pos, ps, P, I)
            assert 0 <= p < P and 0 <= slot < ps // P
            assert (p, page, slot) not in seen
            seen.add((p, page, slot))
            assert oracle.placement_inverse(pages, page, slot, p, ps, P, I) == pos
            assert oracle.placement(pages, pos, ps, P, 1) == oracle.placement(pages, pos, ps, P)
        # each partner's positions, in physical-slot order, are its stripe
        for p in range(P):
            sp = oracle.stripe_positions(ps * len(pages), P, p, I)
            slots = [oracle.placement(pages, int(x), ps, P, I) for x in sp]
            assert all(s[0] == p for s in slots)
            order = [(list(pages).index(s[1]), s[2]) for s in slots]
            assert order == sorted(order)


def pin_merge_interleaved_equals_one(seed=11):
    """Partials over interleaved stripes merge to the P = 1 result too."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = 4, 2, 8
    for m in [1, 5, 33, 100]:
        q = rng.standard_normal((Hq, D))
        K = rng.standard_normal((m, Hkv, D)) * 2
        V = rng.standard_normal((m, Hkv, D))
        O1, L1 = oracle.attention(q, K, V, 0.4)
        for P, I in [(2, 2), (4, 4), (3, 2)]:
            parts = [oracle.stripe_partial(q, K, V, 0.4, P, p, I) for p in range(P)]
            O, L = oracle.merge([o for o, _ in parts], [l for _, l in parts])
            np.testing.assert_allclose(O, O1, atol=1e-12)
            np.testing.assert_allclose(L, L1, atol=1e-12)


def pin_placement_bijection(seed=0):
    """Brute force over every slot of a row's pages: the map is injective, each
    partner page gets page_size // P slots, and the inverse recovers pos."""
    rng = np.random.default_rng(seed)
    for ps, P in [(16, 1), (16, 2), (16, 4), (64, 8), (64, 4), (8, 8)]:
        pages = rng.permutation(40)[:5]
        n = ps * len(pages)
        seen = {}
        per_page = {}
        for pos in range(n):
            p, page, slot = oracle.placement(pages, pos, ps, P)
            assert 0 <= p < P and 0 <= slot < ps // P
            key = (p, page, slot)
            assert key not in seen, "two positions share a slot"
            seen[key] = pos
            per_page[(p, page)] = per_page.get((p, page), 0) + 1
            assert oracle.placement_inverse(pages, page, slot, p, ps, P) == pos
            if P == 1:
                assert (p, slot) == (0, pos % ps)  # P = 1 is the plain paged layout
            assert int(pages[pos // ps]) == page  # page ids stay logical
        assert len(seen) == n
        assert all(c == ps // P for c in per_page.values())
        assert len(per_page) == P * len(pages)


def pin_stripe_positions():
    for L in [0, 1, 5, 37, 100]:
        for P in [1, 2, 4, 8]:
            allp = np.concatenate([oracle.stripe_positions(L, P, p) for p in range(P)])
            assert sorted(allp.tolist()) == list(range(L))
            for p in range(P):
                sp = oracle.stripe_positions(L, P, p)
                assert len(sp) == max(0, (L - p + P - 1) // P)


def pin_pool_image_golden():
    S = 999.0
    pool = np.full((2, 2, 1, 2, 1), S, dtype=np.float32)
    new = np.arange(10, 16, dtype=np.float32).reshape(6, 1, 1)
    img = oracle.expected_pool_image(pool, [1, 0], list(range(6)), new, 4, 2)
    for p, page, slot, val in _rows("pool_image_ps4_P2.txt"):
        want = S if val == "S" else float(val)
        assert img[int(p), int(page), 0, int(slot), 0] == want


def pin_pool_image_sentinel(seed=1):
    """Every written token appears exactly once, at the slot whose inverse is
    its position; everything else keeps the sentinel bits."""
    rng = np.random.default_rng(seed)
    ps, P, H, D = 16, 4, 2, 8
    pages = rng.permutation(10)[:3]
    n = 37
    pool = np.full((P, 10, H, ps // P, D), 0xFFFF, dtype=np.uint16)
    new = rng.integers(0, 0x7F00, size=(n, H, D), dtype=np.uint16)
    pos = rng.permutation(n)
    img = oracle.expected_pool_image(pool, pages, pos, new, ps, P)
    written = np.argwhere(img[..., 0] != 0xFFFF)
    assert len(written) == n * H
    for p, page, h, slot in written:
        lp = oracle.placement_inverse(pages, page, slot, p, ps, P)
        t = int(np.nonzero(pos == lp)[0][0])
        assert np.array_equal(img[p, page, h, slot], new[t, h])


# ---------------------------------------------------------------- attention

def _brute(q, K, V, scale):
    """Explicit loops, direct exp without max shift (small scores only)."""
    Hq, D = q.shape
    m, Hkv, Dv = V.shape
    g = Hq // Hkv
    O = np.zeros((Hq, Dv))
    L = np.full((Hq,), -np.inf)
    for h in range(Hq):
        if m == 0:
            continue
        kh = h // g
        e = []
        for j in range(m):
            s = 0.0
            for d in range(D):
                s += q[h, d] * K[j, kh, d]
            e.append(math.exp(scale * s))
        z = sum(e)
        for d in range(Dv):
            acc = 0.0
            for j in range(m):
                acc += e[j] * V[j, kh, d]
            O[h, d] = acc / z
        L[h] = math.log(z)
    return O, L


def pin_attention_brute(seed=2):
    rng = np.random.default_rng(seed)
    for Hq, Hkv, D, Dv, m in [(4, 1, 8, 8, 5), (4, 2, 6, 4, 7), (8, 8, 5, 5, 1), (6, 3, 4, 3, 0)]:
        q = rng.standard_normal((Hq, D))
        K = rng.standard_normal((m, Hkv, D))
        V = rng.standard_normal((m, Hkv, Dv))
        sc = 0.37
        O, L = oracle.attention(q, K, V, sc)
        Ob, Lb = _brute(q, K, V, sc)
        np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
        if m:
            np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)
        else:
            assert np.all(L == -np.inf) and np.all(O == 0)


def pin_attention_closed_forms(seed=3):
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = 4, 2, 16
    sc = 0.25
    q = rng.standard_normal((Hq, D))
    # one key: output is its value, LSE is its score
    K = rng.standard_normal((1, Hkv, D))
    V = rng.standard_normal((1, Hkv, D))
    O, L = oracle.attention(q, K, V, sc)
    for h in range(Hq):
        kh = h // 2
        np.testing.assert_allclose(O[h], V[0, kh], atol=1e-14)
        np.testing.assert_allclose(L[h], sc * float(np.dot(q[h], K[0, kh])), atol=1e-12)
    # zero query: uniform weights -> mean of values, LSE = ln m
    m = 9
    K = rng.standard_normal((m, Hkv, D)) * 5
    V = rng.standard_normal((m, Hkv, D))
    O, L = oracle.attention(np.zeros((Hq, D)), K, V, sc)
    for h in range(Hq):
        np.testing.assert_allclose(O[h], V[:, h // 2].mean(axis=0), atol=1e-12)
        np.testing.assert_allclose(L[h], math.log(m), atol=1e-12)
    # identical keys: mean of values, LSE = score + ln m
    K = np.repeat(rng.standard_normal((1, Hkv, D)), m, axis=0)
    O, L = oracle.attention(q, K, V, sc)
    for h in range(Hq):
        kh = h // 2
        np.testing.assert_allclose(O[h], V[:, kh].mean(axis=0), atol=1e-12)
        np.testing.assert_allclose(L[h], sc * float(np.dot(q[h], K[0, kh])) + math.log(m), atol=1e-12)
    # the hand-worked example: scores 0 and ln 3, values e0 and e1
    q1 = np.array([[1.0, 0.0]])
    K1 = np.array([[[0.0, 0.0]], [[math.log(3.0), 0.0]]])
    V1 = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    O, L = oracle.attention(q1, K1, V1, 1.0)
    np.testing.assert_allclose(O[0], [0.25, 0.75], atol=1e-15)
    np.testing.assert_allclose(L[0], math.log(4.0), atol=1e-15)


def pin_attention_library(seed=4):
    """torch scaled_dot_product_attention (float64, CPU) on the same data; LSE
    against scipy's logsumexp of the plain scores."""
    torch = pytest.importorskip("torch")
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(seed)
    for Hq, Hkv, D, Dv, m in [(32, 8, 128, 128, 300), (4, 1, 64, 64, 37), (16, 1, 72, 64, 50)]:
        q = rng.standard_normal((Hq, D))
        K = rng.standard_normal((m, Hkv, D))
        V = rng.standard_normal((m, Hkv, Dv))
        sc = 1 / math.sqrt(D)
        O, L = oracle.attention(q, K, V, sc)
        g = Hq // Hkv
        tq = torch.from_numpy(q).reshape(1, Hq, 1, D)
        tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(g, dim=0).unsqueeze(0)
        tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(g, dim=0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=sc)
        np.testing.assert_allclose(O, ref[0, :, 0].numpy(), atol=1e-12)
        for h in range(Hq):
            s = sc * (K[:, h // g] @ q[h])
            np.testing.assert_allclose(L[h], scipy_special.logsumexp(s), atol=1e-12)


# ---------------------------------------------------------------- merge

def pin_merge_golden():
    rows = {r[0]: [float(x) for x in r[1:]] for r in _rows("merge_two_partials.txt")}
    O, L = oracle.merge(np.array([[rows["O_A"]], [rows["O_B"]]]),
                        np.array([[rows["LSE_A"][0]], [math.log(rows["LSE_B_exp"][0])]]))
    np.testing.assert_allclose(O[0], rows["O"], atol=1e-15)
    np.testing.assert_allclose(L[0], math.log(rows["LSE_exp"][0]), atol=1e-15)


def pin_merge_p_way_equals_one(seed=5):
    """P partners attend like one: merging the P stripe partials gives the
    P = 1 result, for P in {1, 2, 4, 8} and lengths incl. ones shorter than P."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = 8, 2, 16
    for m in [1, 3, 7, 8, 50, 129]:
        q = rng.standard_normal((Hq, D))
        K = rng.standard_normal((m, Hkv, D)) * 3
        V = rng.standard_normal((m, Hkv, D))
        O1, L1 = oracle.attention(q, K, V, 0.3)
        for P in [1, 2, 4, 8]:
            parts = [oracle.stripe_partial(q, K, V, 0.3, P, p) for p in range(P)]
            O, L = oracle.merge([o for o, _ in parts], [l for _, l in parts])
            np.testing.assert_allclose(O, O1, atol=1e-12)
            np.testing.assert_allclose(L, L1, atol=1e-12)


def pin_merge_any_split(seed=6):
    """Any split of the keys into disjoint pieces, merged in any order."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = 4, 4, 8
    m = 40
    q = rng.standard_normal((Hq, D))
    K = rng.standard_normal((m, Hkv, D)) * 2
    V = rng.standard_normal((m, Hkv, D))
    O1, L1 = oracle.attention(q, K, V, 0.5)
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, m), size=trial + 1, replace=False))
        pieces = np.split(rng.permutation(m), cuts)
        parts = [oracle.attention(q, K[idx], V[idx], 0.5) for idx in pieces]
        order = rng.permutation(len(parts))
        O, L = oracle.merge([parts[i][0] for i in order], [parts[i][1] for i in order])
        np.testing.assert_allclose(O, O1, atol=1e-12)
        np.testing.assert_allclose(L, L1, atol=1e-12)


def pin_merge_empty():
    """Empty partials (LSE = -inf) drop out; all-empty merges to 0 / -inf."""
    H, Dv = 3, 4
    O_e = np.zeros((H, Dv))
    L_e = np.full((H,), -np.inf)
    O, L = oracle.merge([O_e, O_e], [L_e, L_e])
    assert np.all(O == 0) and np.all(L == -np.inf)
    rng = np.random.default_rng(7)
    O_a = rng.standard_normal((H, Dv))
    L_a = rng.standard_normal(H)
    O, L = oracle.merge([O_e, O_a, O_e], [L_e, L_a, L_e])
    np.testing.assert_allclose(O, O_a, atol=1e-15)
    np.testing.assert_allclose(L, L_a, atol=1e-15)


# ---------------------------------------------------------------- own token + step

def pin_own_token_plus_context(seed=8):
    """Context partials (P stripes over the context) merged with the causal
    own-token partial equal plain causal attention over [context | new]."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, D, P = 8, 2, 16, 4
    for c, n in [(0, 5), (1, 1), (13, 6), (40, 9)]:
        K = rng.standard_normal((c + n, Hkv, D))
        V = rng.standard_normal((c + n, Hkv, D))
        Q = rng.standard_normal((n, Hq, D))
        Oo, Lo = oracle.causal_own_attention(Q, K[c:], V[c:], 0.25)
        for i in range(n):
            parts = [oracle.stripe_partial(Q[i], K[:c], V[:c], 0.25, P, p) for p in range(P)]
            parts.append((Oo[i], Lo[i]))
            O, L = oracle.merge([o for o, _ in parts], [l for _, l in parts])
            Or, Lr = _brute(Q[i], K[: c + i + 1], V[: c + i + 1], 0.25)
            np.testing.assert_allclose(O, Or, atol=1e-12)
            np.testing.assert_allclose(L, Lr, atol=1e-12)


def pin_expected_step_mixed(seed=9):
    """expected_step on a small mixed workload with padding rows: real tokens
    match brute-force causal attention over the row's logical keys; padding
    tokens are exactly 0 / -inf."""
    w = W.mixed_step(seed=seed, n_decode=3, n_extend=2, dec_ctx=(1, 30), ext_new=(2, 5),
                     ext_ctx=(0, 20), padding_spans=[0, 3], token_multiple=16)
    q = oracle.raw_to_f64(w.q)
    k = oracle.raw_to_f64(w.k_seq)
    v = oracle.raw_to_f64(w.v_seq)
    O, L = oracle.expected_step(q, k, v, w.seq_indptr, w.ctx_len, w.new_len, w.qo_indptr,
                                w.num_real_rows, w.num_tokens, w.scale)
    for b in range(w.num_real_rows):
        for i in range(int(w.new_len[b])):
            t = int(w.qo_indptr[b]) + i
            m = int(w.ctx_len[b]) + i + 1
            s0 = int(w.seq_indptr[b])
            Ob, Lb = _brute(q[t], k[s0: s0 + m], v[s0: s0 + m], w.scale)
            np.testing.assert_allclose(O[t], Ob, atol=1e-12)
            np.testing.assert_allclose(L[t], Lb, atol=1e-12)
    first_pad = int(w.qo_indptr[w.num_real_rows])
    assert first_pad < w.num_tokens
    assert np.all(O[first_pad:] == 0) and np.all(L[first_pad:] == -np.inf)


def pin_mla_kv():
    lat = np.arange(2 * 1 * 6, dtype=np.float64).reshape(2, 1, 6)
    K, V = oracle.mla_kv(lat, 4)
    assert K.shape == (2, 1, 6) and V.shape == (2, 1, 4)
    assert np.array_equal(V[1, 0], [6, 7, 8, 9])


def pin_bf16_bits():
    # hand values: 0x3F80 = 1.0, 0xC000 = -2.0, 0x3EAB = 0.333984375, 0x0001 = 2^-133
    got = oracle.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x3EAB, 0x0001], dtype=np.uint16))
    np.testing.assert_array_equal(got, [1.0, -2.0, 0.333984375, 2.0 ** -133])


def pin_e4m3_closed_forms():
    """Values fixed by the E4M3 format: bias 7, 3 mantissa bits, subnormals
    m/8 * 2^-6, largest finite 1.75 * 2^8 = 448, S.1111.111 = NaN."""
    v = oracle.e4m3_value
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0 and oracle.E4M3_MAX == 448.0
    assert v(0x08) == 2.0 ** -6 and v(0x01) == 2.0 ** -9 and v(0x07) == 7 * 2.0 ** -9
    assert v(0x38) == 1.0 and v(0x40) == 2.0 and v(0x30) == 0.5 and v(0x3C) == 1.5 and v(0x77) == 240.0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    assert v(0x00) == 0.0 and v(0x80) == 0.0 and math.copysign(1.0, v(0x80)) == -1.0
    vals = oracle.e4m3_table()[:0x7F]
    assert np.all(np.diff(vals) > 0)  # non-negative finite codes increase with their value


def pin_e4m3_library():
    """Decode of all 256 codes and round-to-nearest-even encode of in-range
    values (random and every midpoint) agree with torch.float8_e4m3fn."""
    torch = pytest.importorskip("torch")
    table = oracle.e4m3_table()
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(lib), np.isnan(table))
    fin = ~np.isnan(table)
    assert np.array_equal(lib[fin], table[fin])
    rng = np.random.default_rng(12)
    pos = table[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([rng.standard_normal(3000) * 40, rng.standard_normal(500) * 0.01, mids, -mids,
                        mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    mine = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, theirs), int((mine != theirs).sum())


def pin_e4m3_rounding_and_saturation():
    enc = oracle.e4m3_encode
    assert enc(1e9) == 0x7E and enc(-1e9) == 0xFE and enc(449.0) == 0x7E and enc(464.0) == 0x7E
    assert enc(float("inf")) == 0x7E and enc(float("nan")) == 0x7F
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A  # midpoints: to the even code
    assert enc(1.0625 * (1 + 1e-6)) == 0x39 and enc(1.1875 * (1 - 1e-6)) == 0x39
    assert enc(2.0 ** -10) == 0x00 and enc(2.0 ** -10 * 1.001) == 0x01  # half the smallest subnormal
    assert enc(-3 * 2.0 ** -10) == 0x82  # -1.5 * 2^-9: tie between codes 1 and 2, to 2
    for c in range(0x7F):
        assert enc(oracle.e4m3_value(c)) == c and enc(oracle.e4m3_value(c | 0x80)) == (c | 0x80)


def pin_e4m3_quantize_error():
    """Quantise -> dequantise stays within half a unit of the last place: 2^-4
    relative for normal codes, 2^-10 * descale absolute below 2^-6 * descale."""
    rng = np.random.default_rng(13)
    x = W.f32_to_bf16_bits(rng.standard_normal(4000).astype(np.float32) * 3)
    xf = oracle.raw_to_f64(x)
    for descale in [0.0123, 0.0625, 1.0]:
        back = oracle.e4m3_dequantize(oracle.e4m3_quantize(x, descale), descale)
        inr = np.abs(xf) <= 448 * descale
        err = np.abs(back - xf)[inr]
        bound = np.maximum(np.abs(xf[inr]) * 2.0 ** -4, 2.0 ** -10 * descale) * (1 + 1e-6)
        assert np.all(err <= bound)
        assert np.all(np.abs(back[~inr]) == 448 * descale)
    # signed zeros keep their sign bit (S.0000.000), next to each other or not
    z = np.array([0x8000, 0x0000, 0x8000, 0x3F80], dtype=np.uint16)  # bf16 -0, +0, -0, 1.0
    assert list(oracle.e4m3_quantize(z, 0.5)) == [0x80, 0x00, 0x80, 0x40]


PINS = [
    pin_e4m3_closed_forms, pin_e4m3_library, pin_e4m3_rounding_and_saturation, pin_e4m3_quantize_error,
    pin_placement_golden, pin_placement_golden_interleaved, pin_placement_bijection,
    pin_placement_bijection_interleaved, pin_merge_interleaved_equals_one, pin_stripe_positions, pin_pool_image_golden,
    pin_pool_image_sentinel, pin_attention_brute, pin_attention_closed_forms,
    pin_attention_library, pin_merge_golden, pin_merge_p_way_equals_one, pin_merge_any_split,
    pin_merge_empty, pin_own_token_plus_context, pin_expected_step_mixed, pin_mla_kv,
    pin_bf16_bits,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin()


# ---------------------------------------------------------------- planted mistakes

def _blocked_placement(page_row, pos, page_size, P, interleave=1):
    # plausible mistake: contiguous blocks per partner instead of striping
    page = int(page_row[pos // page_size])
    off = pos % page_size
    ps_l = page_size // P
    return off // ps_l, page, off % ps_l


def _logical_page_size_placement(page_row, pos, page_size, P, interleave=1):
    # the review's resident-plan bug: offset taken at the logical page size
    page = int(page_row[pos // page_size])
    off = pos % page_size
    return off % P, page, off


def _attention_wrong_head_map(q, K, V, scale):
    # plausible mistake: head h reads KV head h % Hkv instead of h // g
    Hq, Hkv = q.shape[0], K.shape[1]
    O = np.zeros((Hq, V.shape[2]))
    L = np.full((Hq,), -np.inf)
    if K.shape[0] == 0:
        return O, L
    for h in range(Hq):
        kh = h % Hkv
        o, l = _ORIG_ATTENTION(q[h: h + 1], K[:, kh: kh + 1], V[:, kh: kh + 1], scale)
        O[h], L[h] = o[0], l[0]
    return O, L


def _attention_no_scale(q, K, V, scale):
    return _ORIG_ATTENTION(q, K, V, 1.0)


def _merge_wrong_sign(O_parts, LSE_parts):
    O_parts = np.asarray(O_parts, dtype=np.float64)
    LSE_parts = np.asarray(LSE_parts, dtype=np.float64)
    mx = LSE_parts.max(axis=0)
    w = np.exp(mx[None] - LSE_parts)
    z = w.sum(axis=0)
    return (w[..., None] * O_parts).sum(axis=0) / z[:, None], mx + np.log(z)


def _merge_no_renorm(O_parts, LSE_parts):
    O_parts = np.asarray(O_parts, dtype=np.float64)
    LSE_parts = np.asarray(LSE_parts, dtype=np.float64)
    mx = LSE_parts.max(axis=0)
    w = np.exp(LSE_parts - mx[None])
    return (w[..., None] * O_parts).sum(axis=0), mx + np.log(w.sum(axis=0))


def _causal_off_by_one(q_new, k_new, v_new, scale):
    n = q_new.shape[0]
    O = np.zeros((n, q_new.shape[1], v_new.shape[2]))
    L = np.full((n, q_new.shape[1]), -np.inf)
    for i in range(n):
        O[i], L[i] = _ORIG_ATTENTION(q_new[i], k_new[:i], v_new[:i], scale)
    return O, L


_ORIG_ATTENTION = R.attention

def _e4m3_bias_8(code):
    code = int(code) & 0xFF
    e, m = (code >> 3) & 0xF, code & 7
    sign = -1.0 if code & 0x80 else 1.0
    if e == 0xF and m == 7:
        return float("nan")
    return sign * ((m / 8.0) * 2.0 ** -7 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 8))


def _e4m3_ties_away(x, _vals=None):
    x = float(x)
    if x != x:
        return 0x7F
    a = min(abs(x), 448.0)
    vals = [R.e4m3_value(c) for c in range(0x7F)]
    lo = max(c for c in range(0x7F) if vals[c] <= a)
    code = lo if (vals[lo] == a or lo == 0x7E) else (lo if a - vals[lo] < vals[lo + 1] - a else lo + 1)
    return code | (0x80 if np.signbit(x) else 0)


_ORIG_E4M3_ENCODE = R.e4m3_encode


def _e4m3_no_saturation(x, _vals=None):
    return 0x7F if abs(float(x)) > 448.0 else _ORIG_E4M3_ENCODE(x, _vals)


MUTATIONS = {
    "e4m3_exponent_bias_8": ("e4m3_value", _e4m3_bias_8),
    "e4m3_ties_away_from_zero": ("e4m3_encode", _e4m3_ties_away),
    "e4m3_no_saturation": ("e4m3_encode", _e4m3_no_saturation),
    "blocked_placement": ("placement", _blocked_placement),
    "logical_page_size_offset": ("placement", _logical_page_size_placement),
    "wrong_gqa_head_map": ("attention", _attention_wrong_head_map),
    "dropped_scale": ("attention", _attention_no_scale),
    "merge_wrong_sign": ("merge", _merge_wrong_sign),
    "merge_no_renormalise": ("merge", _merge_no_renorm),
    "causal_off_by_one": ("causal_own_attention", _causal_off_by_one),
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(mutation, monkeypatch):
    attr, fn = MUTATIONS[mutation]
    monkeypatch.setattr(R, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {mutation!r} passed every pin"
