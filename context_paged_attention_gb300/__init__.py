"""Context-parallel striped paged attention for GB300 (sm_103a).

The compute lives in ``libcpattn.so`` (CUDA C++, C ABI, declared in
``include/cpattn.h``); ``binding`` marshals torch tensors into that ABI.
Importing this package does not load the library; the first use of a
binding name does, and raises if the library is missing.
"""

_BINDING_NAMES = (
    "PoolDesc", "CpattnError", "cp_kv_write", "cp_paged_attn_partial", "own_token_attn",
    "lse_merge", "workspace_bytes", "library_path", "load_library", "version",
    "DTYPE_BF16", "DTYPE_FP32",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
