"""The C-ABI library loads and exports every declared entry point; host-only
calls (sizes, status strings, argument validation) work without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verification_pass_gb300 import binding
    return binding


def _declared():
    text = open(os.path.join(ROOT, "include", "spec_verify.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    L = lib.lib()
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(lib.EXPORTED)


def test_status_strings(lib):
    L = lib.lib()
    for s in range(0, -7, -1):
        assert L.spec_status_string(s)
    assert L.spec_status_string(-99) == b"unknown status"


def test_sizes(lib):
    c8 = lib.LLAMA_8B
    wb = lib.spec_model_weight_bytes(c8)
    # 32 layers x (6144+4096+28672+14336... ) -- matrices dominate: ~8.03e9 params
    params = 2 * 128256 * 4096 + 32 * (6144 * 4096 + 4096 * 4096 + 2 * 14336 * 4096 + 4096 * 14336)
    assert params * 2 <= wb < params * 2 + 2_000_000   # + fp32 norm gains, alignment
    assert lib.spec_kv_bytes(c8, 1, 2064) == 32 * 1 * 8 * 2064 * 128 * 2
    assert lib.spec_workspace_bytes(c8, 1, 4, 2064) > 0
    bad = lib.ModelConfig(2, 100, 4, 2, 64, 10)      # d not a multiple of 128
    assert lib.spec_model_weight_bytes(bad) == 0
    bad = lib.ModelConfig(2, 256, 4, 3, 64, 10)      # heads not a multiple of kv heads
    assert lib.spec_model_weight_bytes(bad) == 0


def test_argument_validation_without_gpu(lib):
    L = lib.lib()
    P = ctypes.c_void_p
    # NULL pointers are rejected before any CUDA call
    assert L.spec_accept(None, None, None, None, 1, 4, 10, 1.0, 1.0, None, None, None, 0, None) == lib.SPEC_EINVAL
    assert L.spec_draft_sample(None, 1, 10, 1.0, 1.0, None, None, None, None, 0, None) == lib.SPEC_EINVAL
    assert L.spec_verify_forward(None, None, 1, 4, None, None, None, 0, None) == lib.SPEC_EINVAL
    assert L.spec_kv_truncate(None, None, 4, None, None) == lib.SPEC_EINVAL
    # bad temperature / top_p
    fake = P(4096)
    assert L.spec_accept(fake, fake, fake, fake, 1, 4, 10, -1.0, 1.0, fake, fake, fake, 256, None) == lib.SPEC_EINVAL
    assert L.spec_accept(fake, fake, fake, fake, 1, 4, 10, 1.0, 0.0, fake, fake, fake, 256, None) == lib.SPEC_EINVAL
    assert L.spec_accept(fake, fake, fake, fake, 1, 4, 10, 1.0, 1.5, fake, fake, fake, 256, None) == lib.SPEC_EINVAL
    # workspace too small
    assert L.spec_accept(fake, fake, fake, fake, 1, 4, 10, 1.0, 1.0, fake, fake, fake, 8, None) == lib.SPEC_ESIZE
    # zero-size batch is a no-op
    ws0 = lib.spec_accept_workspace_bytes(0, 4, 10)
    assert L.spec_accept(fake, fake, fake, fake, 0, 4, 10, 1.0, 1.0, fake, fake, fake, ws0, None) == lib.SPEC_OK
    # more than 128 rows per sequence, or a misaligned workspace
    big = lib.spec_accept_workspace_bytes(1, 128, 10)
    assert L.spec_accept(fake, fake, fake, fake, 1, 128, 10, 1.0, 1.0, fake, fake, fake, big, None) == lib.SPEC_ESIZE
    ws1 = lib.spec_accept_workspace_bytes(1, 4, 10)
    assert L.spec_accept(fake, fake, fake, fake, 1, 4, 10, 1.0, 1.0, fake, fake, P(4100), ws1, None) == lib.SPEC_EINVAL
    # the accept workspace grows with the batch and the draft length
    assert lib.spec_accept_workspace_bytes(2, 4, 32000) > lib.spec_accept_workspace_bytes(1, 4, 32000)
    assert lib.spec_accept_workspace_bytes(1, 7, 32000) > lib.spec_accept_workspace_bytes(1, 4, 32000)
    out = P()
    cfg = lib.LLAMA_1B.c()
    assert L.spec_model_create(ctypes.byref(cfg), 1, None, 0, None, ctypes.byref(out)) == lib.SPEC_EINVAL
    assert L.spec_model_destroy(None) == lib.SPEC_OK
    # the bounded-wait self-test: a limit outside (0, 2000] ms, a NULL or
    # misaligned pointer, or a workspace below one status word
    assert L.spec_wait_selftest(fake, 1, 0.0, fake, 256, None) == lib.SPEC_EINVAL
    assert L.spec_wait_selftest(fake, 1, 2500.0, fake, 256, None) == lib.SPEC_EINVAL
    assert L.spec_wait_selftest(None, 1, 50.0, fake, 256, None) == lib.SPEC_EINVAL
    assert L.spec_wait_selftest(P(4098), 1, 50.0, fake, 256, None) == lib.SPEC_EINVAL
    assert L.spec_wait_selftest(fake, 1, 50.0, fake, 2, None) == lib.SPEC_EINVAL


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verification_pass_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", src, re.M), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith(".py"):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert "speculative_decoding_verification_pass_gb300" not in src, f


def test_tree_masks_match_the_oracle(lib):
    """spec_tree_masks (host only) gives the oracle's visibility matrix as
    bit masks and its depths, for the pages' tree, chains and random trees;
    malformed trees and trees above 64 nodes are refused."""
    import numpy as np

    from oracle import tree as Tr
    from speculative_decoding_verification_pass_gb300 import workloads as wl

    trees = [Tr.full_tree_parents(2, 2), Tr.full_tree_parents(3, 3), Tr.chain_parents(1),
             Tr.chain_parents(64), [-1, 0, 0, 0, 1, 1, 3, 6, 2]]
    trees += [wl.random_tree(s, n) for s, n in ((1, 5), (2, 33), (3, 64))]
    for par in trees:
        anc, depth = lib.spec_tree_masks(par)
        d_ref, vis = Tr.tree_structure(par)
        n = len(par)
        bits = np.array([[(a >> j) & 1 for j in range(n)] for a in anc])
        np.testing.assert_array_equal(bits, vis)
        assert all(a >> n == 0 for a in anc)
        assert depth == d_ref.tolist()
    for bad in ([0, 0], [-1, 1], [-1, 0, 3, 1], [-1, -1]):
        with pytest.raises(lib.SpecError):
            lib.spec_tree_masks(bad)
    with pytest.raises(lib.SpecError) as e:
        lib.spec_tree_masks(Tr.chain_parents(65))
    assert e.value.status == lib.SPEC_ESIZE
    L = lib.lib()
    fake = ctypes.c_void_p(4096)
    # tree calls validate before touching the device
    assert L.spec_tree_accept(None, None, None, None, None, 1, 4, 10, 1.0, 1.0, None, None, None,
                              None, 0, None) == lib.SPEC_EINVAL
    ws = lib.spec_tree_accept_workspace_bytes(1, 10)
    assert L.spec_tree_accept(fake, fake, fake, fake, fake, 1, 65, 10, 1.0, 1.0, fake, fake, fake,
                              fake, ws, None) == lib.SPEC_ESIZE
    assert L.spec_tree_accept(fake, fake, fake, fake, fake, 1, 4, 10, 1.0, 1.0, fake, fake, fake,
                              fake, ws - 1, None) == lib.SPEC_ESIZE
    assert L.spec_kv_tree_commit(None, None, None, None, 4, None, None) == lib.SPEC_EINVAL
    assert L.spec_verify_forward_tree(None, None, None, None, 1, 4, None, None, None, 0,
                                      None) == lib.SPEC_EINVAL


def test_missing_library_fails_loudly(lib, monkeypatch, tmp_path):
    """Without the built library the binding raises: there is no fallback."""
    from speculative_decoding_verification_pass_gb300 import _build
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "libspec_missing.so"))
    monkeypatch.setattr(lib, "_LIB", None)
    with pytest.raises(RuntimeError, match="not built"):
        lib.lib()
    with pytest.raises(RuntimeError, match="not built"):
        lib.spec_workspace_bytes(lib.LLAMA_8B, 1, 4, 4096)


def test_header_and_library_from_plain_c(lib, tmp_path):
    """include/spec_verify.h compiles as C99 (no C++), the library links from
    C, and the host-only calls behave as documented (tests/c/abi_from_c.c)."""
    import shutil
    import subprocess
    from speculative_decoding_verification_pass_gb300 import _build
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    so = _build.LIB
    exe = str(tmp_path / "abi_from_c")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
                        so, "-Wl,-rpath," + os.path.dirname(so), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
