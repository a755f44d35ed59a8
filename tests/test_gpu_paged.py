"""GPU parity of the paged KV cache.

The paged pass must give the contiguous pass's logits bit for bit when both
caches hold the same rows (pages handed out interleaved across sequences, so
no sequence's pages are contiguous), under the persistent and the per-step
schedules, and agree with the fp64 oracle within |d| <= 1e-2 (1 + |logit|).
After the accept, the device rollback plus the host pool's release must
return exactly the pages past the new length, and the next pass (on pages
taken from the free list again) must still agree.  A page id outside the
pool must be flagged and leave the sequence untouched.
"""
import numpy as np
import pytest
import torch

from oracle import model as OM
from oracle import weights as OW
from speculative_decoding_verification_pass_gb300 import binding as sb
from speculative_decoding_verification_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CFGS = [
    sb.ModelConfig(2, 256, 4, 2, 256, 1000),        # hd 64
    sb.ModelConfig(2, 512, 4, 1, 384, 4099),        # hd 128, 4 query heads per KV head
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _close(got, ref, tol=1e-2):
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert err.max() <= tol, err.max()


def _reserve_interleaved(pk, lens, n, order):
    for b in order:
        pk.reserve(b, int(lens[b]) + n)
    pk.sync()


@pytest.mark.parametrize("schedule", ["persistent", "per_step"])
@pytest.mark.parametrize("ci", range(len(CFGS)))
def test_paged_equals_contiguous_and_oracle(schedule, ci, monkeypatch):
    if schedule == "per_step":
        monkeypatch.setenv("SPEC_FORWARD_PERSISTENT", "0")
    cfg = CFGS[ci]
    B, max_pages = 3, 4
    cap = max_pages * sb.PAGE_SLOTS
    seed = 40 + ci
    m = sb.Model(cfg, seed)
    kc = sb.KVCache(cfg, B, cap)
    pk = sb.PagedKVCache(cfg, B, n_pages=B * max_pages + 3, max_pages=max_pages)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 127, cap))
    ocfg = OM.Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn, cfg.vocab,
                     cfg.rms_eps, cfg.rope_theta)
    W = OW.Weights(ocfg, seed)
    okv = OM.KVState(ocfg, B, cap)
    lens = np.zeros(B, np.int64)
    rng = np.random.default_rng(seed)

    def both(toks):
        n = toks.shape[1]
        _reserve_interleaved(pk, lens, n, rng.permutation(B))
        t = _dev(toks.astype(np.int32))
        a = torch.empty(B, n, cfg.vocab, device="cuda")
        b = torch.empty_like(a)
        sb.spec_verify_forward(m.handle, t, B, n - 1, kc, a, ws)
        sb.spec_verify_forward_paged(m.handle, t, B, n - 1, pk, b, ws)
        assert torch.equal(a, b)
        o = OM.forward(ocfg, W, toks, okv)
        _close(b.double().cpu().numpy(), o)
        lens[:] += n
        return b

    both(wl.tokens(seed, B, 40, cfg.vocab))           # prefill: pages 0..1 of each sequence
    assert (pk.host_table()[:, 0] >= 0).all()
    # rollback: keep 3 / 0 / 5 of a 6-draft pass, then release the pages past the length
    both(wl.tokens(seed, B, 7, cfg.vocab, stream=11))
    keep = np.array([3, 0, 5], np.int32)
    sb.spec_kv_truncate(kc, _dev(keep), 6, ws)
    sb.spec_paged_kv_truncate(pk, _dev(keep), 6, ws)
    okv.lens -= 6 - keep
    lens[:] -= 6 - keep
    free0 = pk.free_pages()
    for b in range(B):
        pk.release(b, int(lens[b]))
    t = pk.host_table()
    for b in range(B):
        np_ = -(-int(lens[b]) // sb.PAGE_SLOTS)
        assert (t[b, :np_] >= 0).all() and (t[b, np_:] == -1).all()
    assert pk.free_pages() >= free0
    np.testing.assert_array_equal(pk.len.cpu().numpy(), lens)
    # a long pass crossing page boundaries, on pages from the free list again
    both(wl.tokens(seed, B, 70, cfg.vocab, stream=12))
    both(wl.tokens(seed, B, 5, cfg.vocab, stream=13))
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    pk.close()


def test_bad_page_is_flagged():
    cfg = CFGS[0]
    B, max_pages = 2, 2
    m = sb.Model(cfg, 3)
    pk = sb.PagedKVCache(cfg, B, n_pages=4, max_pages=max_pages)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 7, max_pages * sb.PAGE_SLOTS))
    pk.reserve(0, 8)
    pk.reserve(1, 8)
    pk.sync()
    pk.table[1, 0] = 4                                # outside the pool
    logits = torch.empty(B, 8, cfg.vocab, device="cuda")
    sb.spec_verify_forward_paged(m.handle, _dev(wl.tokens(3, B, 8, cfg.vocab).astype(np.int32)), B, 7,
                                 pk, logits, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_EDEVICE and bits & sb.DEV_BAD_PAGE
    assert pk.len.cpu().numpy().tolist() == [8, 0]
    pk.close()
