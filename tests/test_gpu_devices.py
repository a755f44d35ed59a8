"""Per-device set-up: kernel attributes (dynamic shared memory limits, cluster
sizes) and occupancy-derived grid sizes are per device in CUDA, so the
library makes each of them once per device.  With two or more GPUs in the
process, the same calls on device 0 and then device 1 must give identical
results; with one GPU the test is skipped.
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


def _run_on(dev, monkeypatch):
    with torch.cuda.device(dev):
        d = f"cuda:{dev}"
        cfg = sb.ModelConfig(2, 512, 4, 1, 384, 4099)
        m = sb.Model(cfg, 5, device=d)
        B, n, cap = 2, 5, 64
        kv = sb.KVCache(cfg, B, cap, device=d)
        ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, n - 1, cap), device=d)
        toks = torch.from_numpy(wl.tokens(6, B, n, cfg.vocab)).to(d)
        z = torch.empty(B, n, cfg.vocab, device=d)
        sb.spec_verify_forward(m.handle, toks, B, n - 1, kv, z, ws)
        head = torch.empty(16, cfg.vocab, device=d)
        hb = torch.from_numpy(wl.hidden_bf16(7, 16, cfg.d_model).view(np.int16)).to(d)
        sb.spec_lm_head(m.handle, hb, 16, head, ws)
        res = [z.cpu(), head.cpu()]
        # both accept schedules: the cooperative grid and one CTA per sequence
        zq, zp = wl.accept_logits(8, B, n - 1, cfg.vocab)
        q = torch.softmax(torch.from_numpy(zq[:, :n - 1]).double(), -1).float().to(d)
        x = torch.from_numpy(wl.tokens(9, B, n - 1, cfg.vocab)).to(d)
        u = torch.from_numpy(wl.uniforms(10, B, n)).to(d)
        aws = sb.workspace(sb.spec_accept_workspace_bytes(B, n - 1, cfg.vocab), device=d)
        for grid in ("1", "0"):
            monkeypatch.setenv("SPEC_ACCEPT_GRID", grid)
            out = torch.empty(B, n, dtype=torch.int32, device=d)
            nacc = torch.empty(B, dtype=torch.int32, device=d)
            sb.spec_accept(torch.from_numpy(zp).to(d), q, x, u, B, n - 1, cfg.vocab, 1.0, 0.9,
                           out, nacc, aws)
            res += [out.cpu(), nacc.cpu()]
        torch.cuda.synchronize(dev)
        assert sb.spec_device_status(ws)[0] == sb.SPEC_OK
        assert sb.spec_device_status(aws)[0] == sb.SPEC_OK
        m.close()
        return res


def test_second_device_gives_the_same_results(monkeypatch):
    if torch.cuda.device_count() < 2:
        pytest.skip("one GPU in this process")
    a = _run_on(0, monkeypatch)
    b = _run_on(1, monkeypatch)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
