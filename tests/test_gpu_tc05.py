"""Tensor-core plumbing self-test (cpattn_umma_selftest) against a plain matmul.

Checks the shared-memory operand layouts, tcgen05 descriptors, TMEM
allocation and read-back the attention kernels are built on: the Q K^T
pattern (both operands K-major, 128-byte swizzle) and the P V pattern
(64-byte-swizzled K-major A, 128-byte-swizzled rows read M/N-major as B).
Exchanging the two descriptor strides of the M/N-major operand must change
the result, which pins which field carries which stride.
"""

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def selftest():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from context_paged_attention_gb300 import binding as B

    f = B.load_library().cpattn_umma_selftest
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p]
    return f


def _run(f, variant, N, K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    qk = variant in (0, 4)  # D = A B^T with B [N][K]; else D = A B with A [128][32]
    A = torch.randn(128, K if qk else 32, device="cuda", generator=g).bfloat16()
    if qk:
        Bm = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    else:
        Bm = torch.randn(32, N, device="cuda", generator=g).bfloat16()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = f(variant, A.data_ptr(), Bm.data_ptr(), D.data_ptr(), N, K, st.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 0
    ref = A.double() @ (Bm.double().t() if qk else Bm.double())
    return float((D.double() - ref).abs().max())


@pytest.mark.parametrize("N,K", [(16, 64), (32, 128), (128, 192), (256, 256)])
def test_qk_pattern(selftest, N, K):
    # fp32 accumulation of K exact bf16 products
    assert _run(selftest, 0, N, K, seed=N + K) <= 1e-3


@pytest.mark.parametrize("N", [64, 128, 256])
def test_pv_pattern(selftest, N):
    assert _run(selftest, 1, N, 32, seed=N) <= 1e-3


def test_exchanged_strides_differ(selftest):
    assert _run(selftest, 2, 256, 32, seed=3) > 1.0


def test_shapes_beyond_the_tile_are_refused(selftest):
    x = torch.zeros(16, device="cuda")
    assert selftest(0, x.data_ptr(), x.data_ptr(), x.data_ptr(), 272, 64, None, None) == -3
    assert selftest(1, x.data_ptr(), x.data_ptr(), x.data_ptr(), 256, 64, None, None) == -3


@pytest.mark.parametrize("N", [64, 128, 256])
def test_pv_pattern_a_in_tmem(selftest, N):
    # P V with P in tensor memory (row m in lane m, bf16 pairs a column): the
    # layout a kernel keeping P in TMEM relies on
    assert _run(selftest, 3, N, 32, seed=N + 7) <= 1e-3


@pytest.mark.parametrize("N,K", [(32, 128), (128, 192), (256, 256)])
def test_qk_pattern_a_in_tmem(selftest, N, K):
    # Q K^T with Q in tensor memory over several k-steps
    assert _run(selftest, 4, N, K, seed=N + K + 11) <= 1e-3


def test_bounded_wait_times_out_and_frees(selftest):
    # a completion barrier nobody arrives at: the bounded wait gives up, the
    # call reports CPATTN_DEV_TC_TIMEOUT (4), frees its tensor memory, and the
    # next tensor-core call on the same stream allocates and runs normally
    x = torch.zeros(16, device="cuda", dtype=torch.bfloat16)
    D = torch.full((128, 16), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        st.zero_()
        rc = selftest(5, x.data_ptr(), x.data_ptr(), D.data_ptr(), 0, 0, st.data_ptr(), stream)
        torch.cuda.synchronize()
        assert rc == 0 and int(st.item()) == 4
        assert torch.isnan(D).all()  # the timed-out call wrote nothing
    assert _run(selftest, 0, 128, 128, seed=5) <= 1e-3
    assert _run(selftest, 4, 256, 256, seed=6) <= 1e-3  # 512 TMEM columns: all of it was freed
