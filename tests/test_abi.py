"""The C-ABI library: it builds, loads, exports every declared symbol, and its
host-side argument checks return the documented status codes (no GPU needed:
every call here fails validation before anything is launched)."""

import ctypes
import os
import re

import pytest

from context_paged_attention_gb300 import binding as B
from context_paged_attention_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return B.load_library()


def declared_functions():
    text = ""
    for name in sorted(os.listdir(os.path.dirname(HEADER))):
        if name.endswith(".h"):
            text += open(os.path.join(os.path.dirname(HEADER), name)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:CPATTN_API\s+)?(?:int|size_t|const char\s*\*)\s+(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ["cp_kv_write", "cp_paged_attn_partial", "own_token_attn", "lse_merge",
              "cp_paged_attn_workspace_bytes", "cpattn_version", "cpattn_status_string", "cpattn_pool_bytes"]:
        assert n in names, n


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in cpattn.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.cpattn_version() == 3
    assert lib.cpattn_status_string(0) == b"ok"
    assert b"divide" in lib.cpattn_status_string(-2)
    assert lib.cpattn_status_string(-999) == b"unknown status"


def _desc(**kw):
    d = dict(P=4, page_size=16, num_pages=10, num_kv_heads=8, head_dim=128, head_dim_v=128, dtype=B.DTYPE_BF16)
    d.update(kw)
    return B.PoolDesc(**d)


FAKE = 0x10000  # never dereferenced: these calls fail host validation first


def test_pool_bytes(lib):
    d = _desc()
    assert lib.cpattn_pool_bytes(ctypes.byref(d), 0) == 4 * 10 * 8 * 4 * 128 * 2
    mla = _desc(num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64)
    assert lib.cpattn_pool_bytes(ctypes.byref(mla), 0) == 4 * 10 * 1 * 16 * 576 * 2
    assert lib.cpattn_pool_bytes(ctypes.byref(_desc(P=3)), 0) == 0


@pytest.mark.parametrize("P,ps", [(3, 16), (0, 16), (32, 16), (-1, 8)])
def test_p_must_divide_page_size(lib, P, ps):
    d = _desc(P=P, page_size=ps)
    st = lib.cp_kv_write(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None)
    assert st == -2
    st = lib.cp_paged_attn_partial(ctypes.byref(d), FAKE, FAKE, FAKE, 32, 1, 1, None, FAKE, 100, FAKE, FAKE, 0.1,
                                   FAKE, FAKE, FAKE, 1 << 30, None, None)
    assert st == -2


@pytest.mark.parametrize("I", [3, -1, 8, 5])
def test_interleave_times_p_must_divide_page_size(lib, I):
    d = _desc(interleave=I)  # P 4, page 16: I in {0, 1, 2, 4} only
    st = lib.cp_kv_write(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None)
    assert st == -2
    assert lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 256) == 0
    assert lib.cpattn_pool_bytes(ctypes.byref(d), 0) == 0


@pytest.mark.parametrize("I", [0, 1, 2, 4])
def test_interleave_accepted(lib, I):
    d = _desc(interleave=I)
    assert lib.cpattn_pool_bytes(ctypes.byref(d), 0) == 4 * 10 * 8 * 4 * 128 * 2
    assert lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 8192) > 0


def test_invalid_and_misaligned(lib):
    d = _desc()
    # null pool
    assert lib.cp_kv_write(ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, FAKE, FAKE, None, None) == -1
    # misaligned k_new
    assert lib.cp_kv_write(ctypes.byref(d), FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, 1, 1, FAKE, FAKE, None,
                           None) == -4
    # MLA pools take no V
    mla = _desc(num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64)
    assert lib.cp_kv_write(ctypes.byref(mla), FAKE, FAKE, FAKE, None, FAKE, FAKE, 1, 1, FAKE, FAKE, None,
                           None) == -1
    # query heads not a multiple of KV heads
    assert lib.cp_paged_attn_partial(ctypes.byref(d), FAKE, FAKE, FAKE, 30, 1, 1, None, FAKE, 100, FAKE, FAKE, 0.1,
                                     FAKE, FAKE, FAKE, 1 << 30, None, None) == -1
    # one token a row needs num_tokens == num_rows when qo_indptr is NULL
    assert lib.cp_paged_attn_partial(ctypes.byref(d), FAKE, FAKE, FAKE, 32, 2, 3, None, FAKE, 100, FAKE, FAKE, 0.1,
                                     FAKE, FAKE, FAKE, 1 << 30, None, None) == -1
    # head_dim_v above head_dim, and rows that are not 16-byte multiples
    assert lib.cp_paged_attn_partial(ctypes.byref(_desc(head_dim_v=256)), FAKE, FAKE, FAKE, 32, 1, 1, None, FAKE,
                                     100, FAKE, FAKE, 0.1, FAKE, FAKE, FAKE, 1 << 30, None, None) == -3
    assert lib.cp_paged_attn_partial(ctypes.byref(_desc(head_dim=4, head_dim_v=4)), FAKE, FAKE, FAKE, 32, 1, 1,
                                     None, FAKE, 100, FAKE, FAKE, 0.1, FAKE, FAKE, FAKE, 1 << 30, None, None) == -3
    # multi-token rows over a bf16 pool of 2^31 or more K rows: refused before any launch
    huge = _desc(num_pages=1 << 26)  # 2^26 pages x 8 heads x 16 slots = 2^33 rows
    assert lib.cp_paged_attn_partial(ctypes.byref(huge), FAKE, FAKE, FAKE, 32, 2, 8, FAKE, FAKE, 100, FAKE, FAKE,
                                     0.1, FAKE, FAKE, FAKE, 1 << 30, None, None) == -3
    # merge: bad counts / dims
    assert lib.lse_merge(0, FAKE, FAKE, 0, 0, 1, 1, 128, 0, FAKE, None, None) == -1
    assert lib.lse_merge(2, FAKE, FAKE, 10, 1, 1, 1, 128, 0, FAKE, None, None) == -1
    assert lib.lse_merge(1, FAKE, FAKE, 0, 0, 1, 1, 6, 0, FAKE, None, None) == -1
    # own-token: real rows beyond the bucket
    assert lib.own_token_attn(FAKE, FAKE, FAKE, 32, 8, 128, 128, 0, FAKE, 4, 5, 16, 8, 0.1, FAKE, FAKE,
                              None) == -1


def test_fp8_descriptor_checks(lib):
    fp8 = dict(kv_dtype=2, k_descale=0.0123, v_descale=0.0137)
    d = _desc(**fp8)
    assert lib.cpattn_pool_bytes(ctypes.byref(d), 0) == 4 * 10 * 8 * 4 * 128  # one byte a code
    assert lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 8192) > 0
    # FP8 pools belong to bf16 layers; descales must be finite and positive
    assert lib.cpattn_pool_bytes(ctypes.byref(_desc(dtype=B.DTYPE_FP32, **fp8)), 0) == 0
    for ks in [0.0, -1.0, float("nan"), float("inf")]:
        bad = _desc(kv_dtype=2, k_descale=ks, v_descale=0.5)
        assert lib.cp_kv_write(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, FAKE, FAKE, None,
                               None) == -1
    # an unknown pool type, and a pool type other than the layer's that is not FP8
    assert lib.cpattn_pool_bytes(ctypes.byref(_desc(kv_dtype=7)), 0) == 0
    assert lib.cpattn_pool_bytes(ctypes.byref(_desc(kv_dtype=1)), 0) == 0
    # kv_dtype 0 and kv_dtype == dtype mean the same pool
    assert lib.cpattn_pool_bytes(ctypes.byref(_desc(kv_dtype=0)), 0) == \
        lib.cpattn_pool_bytes(ctypes.byref(_desc(kv_dtype=B.DTYPE_BF16)), 0)
    # E4M3 pools are for GQA layers: an MLA descriptor is refused before any launch
    mla = _desc(num_kv_heads=1, head_dim=576, head_dim_v=512, page_size=64, **fp8)
    assert lib.cp_paged_attn_partial(ctypes.byref(mla), FAKE, FAKE, FAKE, 128, 1, 1, None, FAKE, 100, FAKE, FAKE,
                                     0.1, FAKE, FAKE, FAKE, 1 << 30, None, None) == -3


def test_fused_argument_checks(lib):
    d = _desc()
    args = lambda extra_o, extra_lse, odt, out: (ctypes.byref(d), FAKE, FAKE, FAKE, 32, 1, 1, None, FAKE, 100, FAKE,
                                                 FAKE, None, 0.1, extra_o, extra_lse, odt, out, None, FAKE, 1 << 30,
                                                 None, None)
    assert lib.cp_paged_attn_fused(*args(None, None, 7, FAKE)) == -1           # unknown output type
    assert lib.cp_paged_attn_fused(*args(FAKE, None, 0, FAKE)) == -1           # extra partial half given
    assert lib.cp_paged_attn_fused(*args(None, None, 0, None)) == -1           # no output
    assert lib.cp_paged_attn_fused(*args(None, None, 0, FAKE + 8)) == -4       # misaligned output
    bad = _desc(P=3)
    assert lib.cp_paged_attn_fused(ctypes.byref(bad), FAKE, FAKE, FAKE, 32, 1, 1, None, FAKE, 100, FAKE, FAKE, None,
                                   0.1, None, None, 0, FAKE, None, FAKE, 1 << 30, None, None) == -2
    # workspace: always room for every chunk partial (the split path may need none)
    fused = lib.cp_paged_attn_fused_workspace_bytes(ctypes.byref(d), 32, 64, 256)
    plain = lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 256)
    assert fused >= 64 * 4 * 32 * 128 * 4 and fused > plain
    assert lib.cp_paged_attn_fused(ctypes.byref(d), FAKE, FAKE, FAKE, 32, 64, 64, None, FAKE, 256, FAKE, FAKE, None,
                                   0.1, None, None, 0, FAKE, None, FAKE, fused - 1, None, None) == -5


def test_partial_ex_and_view_checks(lib):
    d = _desc()
    # LSE layouts 0 (token-major) and 1 (head-major) only
    assert lib.cp_paged_attn_partial_ex(ctypes.byref(d), FAKE, FAKE, FAKE, 32, 1, 1, None, FAKE, 100, FAKE, FAKE,
                                        0.1, FAKE, FAKE, 2, None, FAKE, 1 << 30, None, None) == -1
    V = B.PartialView
    good = V(FAKE, FAKE, 512, 128, 4, 1)
    arr = (V * 17)(*([good] * 17))
    assert lib.lse_merge_views(0, arr, 4, 4, 128, 0, FAKE, 512, 128, None, 0, 0, None) == -1
    assert lib.lse_merge_views(17, arr, 4, 4, 128, 0, FAKE, 512, 128, None, 0, 0, None) == -1  # > 16 views
    assert lib.lse_merge_views(1, arr, 4, 4, 126, 0, FAKE, 512, 128, None, 0, 0, None) == -1  # dv % 4
    assert lib.lse_merge_views(1, arr, 4, 4, 128, 5, FAKE, 512, 128, None, 0, 0, None) == -1  # out type
    bad = (V * 1)(V(FAKE + 4, FAKE, 512, 128, 4, 1))
    assert lib.lse_merge_views(1, bad, 4, 4, 128, 0, FAKE, 512, 128, None, 0, 0, None) == -4  # row not 16-B aligned
    bad = (V * 1)(V(FAKE, FAKE, 514, 128, 4, 1))
    assert lib.lse_merge_views(1, bad, 4, 4, 128, 0, FAKE, 512, 128, None, 0, 0, None) == -4  # stride
    assert lib.lse_merge_views(1, arr, 4, 4, 128, 0, FAKE, 510, 128, None, 0, 0, None) == -4  # out stride
    nul = (V * 1)(V(FAKE, None, 512, 128, 4, 1))
    assert lib.lse_merge_views(1, nul, 4, 4, 128, 0, FAKE, 512, 128, None, 0, 0, None) == -1
    assert lib.lse_merge_views(1, arr, 0, 4, 128, 0, FAKE, 512, 128, None, 0, 0, None) == 0  # nothing to do


def test_workspace_sizing(lib):
    d = _desc()
    small = lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 256)
    mid = lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 8192)
    # stripes past one split-KV chunk need room for the chunk partials
    big = lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 32, 64, 1 << 16)
    assert small > 0 and mid >= small and big > mid
    assert lib.cp_paged_attn_workspace_bytes(ctypes.byref(d), 30, 64, 8192) == 0
    # too-small workspace is refused before any launch
    assert lib.cp_paged_attn_partial(ctypes.byref(d), FAKE, FAKE, FAKE, 32, 64, 64, None, FAKE, 8192, FAKE, FAKE,
                                     0.1, FAKE, FAKE, FAKE, mid - 1, None, None) == -5
    assert lib.cp_paged_attn_partial(ctypes.byref(d), FAKE, FAKE, FAKE, 32, 64, 64, None, FAKE, 1 << 16, FAKE,
                                     FAKE, 0.1, FAKE, FAKE, FAKE, big - 1, None, None) == -5


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros(4)
    with pytest.raises(ValueError):
        B._ptr(x)


def test_missing_library_is_loud(tmp_path):
    with pytest.raises(RuntimeError):
        B.load_library(str(tmp_path / "nope.so"))
