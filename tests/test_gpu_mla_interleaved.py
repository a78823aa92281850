"""MLA partials stay bit-identical when other kernels run between the calls.

Each call of the MLA kernel starts on SMs whose shared and tensor memory hold
whatever the previous kernels left there, and its warps run at whatever pace
those leftovers and the memory system allow.  A barrier wait that could pass
a phase early (a waiter that skips phases of a parity barrier) shows here as
rows that differ from one call to the next: NaN or stale values of single
warps' rows.  The GQA partial of a mixed step, a GQA decode partial and the
fused MLA call run in turn between the checked calls; every result must equal
the first one bit for bit (the same plan on the same inputs).
"""

import pytest
import torch

from context_paged_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROUNDS = 48


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _att(w):
    from context_paged_attention_gb300.step import StripedAttention

    return StripedAttention(w, device="cuda")


def test_mla_partials_repeat_exactly_between_other_kernels():
    # per-partner stripes cut into pieces (ticket merges) and a fused call over cut tokens
    w = W.mla_decode(seed=44, batch=2, len_lo=2000, len_hi=9000)
    att = _att(w)
    att.write_new()
    fused = _att(W.mla_decode(seed=49, batch=8, len_lo=3000, len_hi=20000))
    fused.write_new()
    others = [_att(W.mixed_step(seed=5, n_decode=12, n_extend=6, token_multiple=64)),
              _att(W.gqa_decode(seed=2, batch=16))]
    att.partial()
    fused.fused()
    torch.cuda.synchronize()
    ref = att.o_parts[: w.P].clone()
    ref_lse = att.lse_parts[: w.P].clone()
    ref_fused = fused.out.clone()
    for r in range(ROUNDS):
        others[r % 2].partial()
        if r % 3 == 0:
            fused.out.fill_(float("nan"))
            fused.fused()
        att.o_parts.fill_(float("nan"))
        att.partial()
        torch.cuda.synchronize()
        assert att.status() == 0 and fused.status() == 0
        bad = torch.nonzero((att.o_parts[: w.P].view(torch.int32) != ref.view(torch.int32)).any(-1))
        assert bad.shape[0] == 0, f"round {r}: {bad.shape[0]} (partner, token, head) rows differ, e.g. {bad[:4].tolist()}"
        assert torch.equal(att.lse_parts[: w.P].view(torch.int32), ref_lse.view(torch.int32)), f"round {r}: LSEs differ"
        if r % 3 == 0:
            assert torch.equal(fused.out.view(torch.int16), ref_fused.view(torch.int16)), f"round {r}: fused output differs"
