"""Host-side checks of the seeded input generator (no GPU, no oracle arithmetic)."""

import math

import numpy as np
import pytest

from context_paged_attention_gb300 import workloads as W


def _check_common(w):
    B = w.num_rows
    assert w.kv_page_indptr.shape == (B + 1,)
    assert w.qo_indptr.shape == (B + 1,)
    assert w.page_size % w.P == 0
    idx = w.kv_page_indices
    assert idx.min() >= 0 and idx.max() < w.num_pages
    real = []
    for b in range(B):
        pages = idx[w.kv_page_indptr[b]: w.kv_page_indptr[b + 1]]
        if b < w.num_real_rows:
            L = int(w.ctx_len[b] + w.new_len[b])
            assert len(pages) == math.ceil(L / w.page_size)
            assert w.sink_page not in pages
            real.extend(pages.tolist())
        else:
            assert np.all(pages == w.sink_page)
    assert len(real) == len(set(real)), "rows share a page"
    # positions: new tokens follow the context, padding tokens are -1
    for b in range(w.num_real_rows):
        span = w.positions[w.qo_indptr[b]: w.qo_indptr[b + 1]]
        assert np.array_equal(span, np.arange(w.ctx_len[b], w.ctx_len[b] + w.new_len[b]))
    assert np.all(w.positions[w.qo_indptr[w.num_real_rows]:] == -1)
    assert w.num_tokens >= w.qo_indptr[-1]


def test_tiny():
    w = W.tiny_fp32()
    _check_common(w)
    assert w.num_pages == 32 and w.P == 2 and w.head_dim == 64 and w.scale == 1 / 8
    assert list(w.ctx_len + w.new_len) == [37, 100]
    assert [int(w.kv_page_indptr[i + 1] - w.kv_page_indptr[i]) for i in range(2)] == [3, 7]
    assert w.q.dtype == np.float32


@pytest.mark.parametrize("fn,kw", [
    (W.gqa_decode, dict(batch=6, len_lo=20, len_hi=300)),
    (W.long_gqa_decode, dict(batch=2, len_lo=500, len_hi=900)),
    (W.mla_decode, dict(batch=3, len_lo=70, len_hi=200)),
    (W.mixed_step, dict(n_decode=4, n_extend=3, dec_ctx=(10, 90), ext_new=(2, 20), ext_ctx=(0, 50),
                        padding_spans=[0, 2, 0], token_multiple=32)),
])
def test_small_variants(fn, kw):
    w = fn(**kw)
    _check_common(w)
    assert w.q.dtype == np.uint16
    # padding queries / new K are NaN bits
    t0 = int(w.qo_indptr[w.num_real_rows])
    if t0 < w.num_tokens:
        assert np.all(w.q[t0:] == W.BF16_NAN)
        assert np.all(w.k_new[t0:] == W.BF16_NAN)
    # same seed -> same draw
    w2 = fn(**kw)
    assert np.array_equal(w.q, w2.q) and np.array_equal(w.kv_page_indices, w2.kv_page_indices)


def test_bf16_rounding_hand_values():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3], dtype=np.float32)
    # 1.00390625 = 1 + 2^-8 is a tie between 0x3F80 and 0x3F81 -> even (0x3F80)
    # 1.005859375 = 1 + 1.5 * 2^-8 rounds up to 0x3F81 (1.0078125)
    bits = W.f32_to_bf16_bits(x)
    assert bits.tolist()[:4] == [0x3F80, 0x3F80, 0x3F81, 0xC020]


def test_full_size_geometry_cheap():
    """Lengths and pool sizes of the full-size workloads (values not drawn here)."""
    rng = np.random.default_rng(2)
    L = rng.integers(512, 8192, size=64, endpoint=True)
    assert L.min() >= 512 and L.max() <= 8192


def test_fp8_pool_bytes_halve():
    w = W.gqa_decode(seed=5, batch=3, len_lo=10, len_hi=100)
    f = W.fp8_pool(w, 0.01, 0.02)
    assert f.kv_bytes_read() * 2 == w.kv_bytes_read() and f.kv_dtype == "fp8" and f.name.endswith("_fp8")
