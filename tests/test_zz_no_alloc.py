"""The LM head that keeps its scratch inside the library.

For callers that cannot allocate device memory (the host owns every
allocation and passes only inputs and outputs).  Checked through the C ABI
against spec_lm_head, which takes a caller workspace, on two calls in a row
(the second call starts from the first call's leftover scratch).  This file
sorts last so that a failure here does not stop the other GPU tests.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_pass_gb300 import binding as sb
from speculative_decoding_verification_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_noalloc_lm_head_matches_workspace_version_twice():
    cfg = sb.ModelConfig(0, 4096, 32, 8, 128, 32000)
    m = sb.Model(cfg, 41)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, 16, 0, 1))
    for call, rows in enumerate((5, 16)):
        hb = torch.from_numpy(wl.hidden_bf16(100 + call, rows, cfg.d_model).view(np.int16)).cuda()
        ref = torch.empty(rows, cfg.vocab, device="cuda")
        got = torch.full((rows, cfg.vocab), float("nan"), device="cuda")
        sb.spec_lm_head(m.handle, hb, rows, ref, ws)
        sb.spec_lm_head_noalloc(m.handle, hb, rows, got)
        torch.cuda.synchronize()
        np.testing.assert_allclose(got.cpu().numpy(), ref.cpu().numpy(), rtol=1e-5, atol=1e-5)
    # limits are reported, not overrun
    big = torch.zeros(17, cfg.d_model, dtype=torch.int16, device="cuda")
    out = torch.empty(17, cfg.vocab, device="cuda")
    with pytest.raises(sb.SpecError):
        sb.spec_lm_head_noalloc(m.handle, big, 17, out)
    m.close()
