"""cp_paged_attn_partial_noalloc: the partner-partial call for callers that
cannot allocate device memory (it uses the library's own fixed scratch array
instead of a caller workspace).  Checked through the C ABI against
cp_paged_attn_partial with a caller workspace, on two calls in a row.  Both
calls run the same kernels with the same plan on the same inputs, and every
split-KV merge combines its chunks in chunk order, so the results must be
identical bit for bit: any stale byte read from the shared array would show.

This file is collected last on purpose (a run that stops at the first failure
has run everything else first); it builds the library itself, so it also runs
alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from context_paged_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from context_paged_attention_gb300 import binding as B

    lib = B.load_library()
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn = lib.cp_paged_attn_partial_noalloc
    fn.restype = i32
    fn.argtypes = [ctypes.POINTER(B.PoolDesc), vp, vp, vp, i32, i32, i32, vp, vp, i32, vp, vp, ctypes.c_float,
                   vp, vp, vp, vp]
    lib.cp_paged_attn_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.cp_paged_attn_noalloc_scratch_bytes.argtypes = []
    return lib


def _noalloc_call(lib, att, o_part, lse_part):
    w = att.w
    stream = torch.cuda.current_stream().cuda_stream
    return lib.cp_paged_attn_partial_noalloc(
        ctypes.byref(att.desc), att.pool_k.data_ptr(), None if att.pool_v is None else att.pool_v.data_ptr(),
        att.q.data_ptr(), w.num_q_heads, w.num_rows, w.num_tokens, att.qo_indptr.data_ptr(),
        att.kv_len.data_ptr(), att.max_kv_len, att.page_indptr.data_ptr(), att.page_indices.data_ptr(),
        w.scale, o_part.data_ptr(), lse_part.data_ptr(), att.dev_status.data_ptr(), stream)


CASES = {
    # stripes of up to 5000 keys: several 2048-key split-KV chunks, so the
    # shared array holds chunk partials and the split tickets are used
    "gqa_decode_split": lambda: W.gqa_decode(seed=41, batch=4, len_lo=12000, len_hi=20000),
    # extend rows whose context stripes split too
    "mixed_step_split": lambda: W.mixed_step(seed=42, n_decode=2, n_extend=2, dec_ctx=(100, 4000),
                                             ext_new=(2, 12), ext_ctx=(9000, 12000), padding_spans=[0, 2],
                                             token_multiple=32),
    # short stripes: no split, the array is not touched
    "gqa_decode": lambda: W.gqa_decode(seed=43, batch=8, len_lo=100, len_hi=6000),
    "mla_decode": lambda: W.mla_decode(seed=44, batch=2, len_lo=2000, len_hi=9000),
}
# cases whose plan must split a stripe (checked below through the workspace size)
SPLITS = {"gqa_decode_split", "mixed_step_split"}


def _same(a, b):
    """Bit-identical float tensors (-inf equal to -inf)."""
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_workspace_call_twice(lib, name):
    from context_paged_attention_gb300.step import StripedAttention

    from context_paged_attention_gb300 import binding as B

    w = CASES[name]()
    att = StripedAttention(w, device="cuda")
    ws = B.workspace_bytes(att.desc, w.num_q_heads, w.num_tokens, att.max_kv_len)
    assert 0 < ws <= lib.cp_paged_attn_noalloc_scratch_bytes()
    if name in SPLITS:
        # more than the tickets alone: chunk partials live in the scratch
        tickets = w.num_tokens * w.P * w.num_kv_heads * 4
        assert ws > 2 * tickets + 1024, "the plan does not split a stripe"
    att.write_new()
    att.partial()  # the existing entry point with a caller workspace
    torch.cuda.synchronize()
    ref_o = att.o_parts[: w.P].clone()
    ref_l = att.lse_parts[: w.P].clone()
    for call in range(2):
        o = torch.full_like(ref_o, float("nan"))
        l = torch.full_like(ref_l, float("nan"))
        st = _noalloc_call(lib, att, o, l)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert att.status() == 0
        assert _same(o, ref_o), f"call {call}: outputs differ from the workspace call"
        assert _same(l, ref_l), f"call {call}: LSEs differ from the workspace call"


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    from context_paged_attention_gb300 import binding as B

    cap = lib.cp_paged_attn_noalloc_scratch_bytes()
    assert cap == 16 << 20
    desc = B.PoolDesc(P=4, page_size=16, num_pages=10, num_kv_heads=8, head_dim=128, head_dim_v=128,
                      dtype=B.DTYPE_BF16)
    # 64 rows of up to 512k keys need far more split scratch than the fixed array
    assert B.workspace_bytes(desc, 32, 64, 1 << 19) > cap
    st = lib.cp_paged_attn_partial_noalloc(ctypes.byref(desc), 0x10000, 0x10000, 0x10000, 32, 64, 64, None,
                                           0x10000, 1 << 19, 0x10000, 0x10000, 0.1, 0x10000, 0x10000, None, None)
    assert st == -5  # CPATTN_ERR_WORKSPACE_TOO_SMALL, nothing launched
