"""CPU-side checks of the C boundary: the library builds, loads without a
GPU, exports every entry point declared in include/*.h, and rejects bad
arguments synchronously (before any device work)."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

import speculative_decoding_draft_sampling_gb300 as sv


@pytest.fixture(scope="module")
def lib():
    sv.build()
    return sv.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(spec_[a-z_0-9]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_tuning(lib):
    assert sv.version() >= 100
    sv.set_tuning(0, 0)
    assert lib.spec_set_tuning(-1, 0) == 1
    assert b"slices_per_row" in lib.spec_last_error()
    sv.set_tuning(0, 0)


def test_workspace_sizes(lib):
    # chain / greedy / tree-walk scratch is one control block whatever the
    # shape; the tree build keeps per-request enumeration state
    a = lib.spec_verify_chain_workspace_size(4, 4, 1000, 0)
    b = lib.spec_verify_chain_workspace_size(256, 8, 151936, 50)
    assert 0 < a <= b <= 4096
    assert 0 < lib.spec_tree_build_workspace_size(4, 16, 151936, 64) < lib.spec_tree_build_workspace_size(32, 16, 151936, 64)
    assert lib.spec_tree_build_workspace_size(32, 17, 151936, 64) == 0      # L > 16 unsupported
    assert lib.spec_tree_build_workspace_size(32, 16, 151936, 257) == 0     # budget > 256
    assert lib.spec_verify_greedy_workspace_size(-1, 3, 10) == 0


def _chain(lib, **kw):
    args = dict(logits=1, ldt=0, lbs=0, lrs=10, q=1, qbs=0, qrs=10, draft=1, u=1, B=2, K=1, V=10,
                T=1.0, top_k=0, kp=None, lo=None, qo=None, tok=1, n=1, st=1, diag=None, ws=16, wsb=1 << 30,
                stream=None)
    args.update(kw)
    return lib.spec_verify_chain(*[args[k] for k in ("logits", "ldt", "lbs", "lrs", "q", "qbs", "qrs", "draft",
                                                     "u", "B", "K", "V", "T", "top_k", "kp", "lo", "qo", "tok",
                                                     "n", "st", "diag", "ws", "wsb", "stream")])


def test_invalid_arguments_rejected_on_host(lib):
    assert _chain(lib, B=-1) == 1
    assert _chain(lib, V=0) == 1
    assert _chain(lib, T=0.0) == 1
    assert _chain(lib, T=float("nan")) == 1
    assert _chain(lib, ldt=7) == 1
    assert _chain(lib, lo=16) == 1                         # row offsets need k_per_req and q offsets
    assert _chain(lib, kp=16, lo=16) == 1
    assert _chain(lib, logits=None) == 1
    assert _chain(lib, lrs=5) == 1                         # row stride < V
    assert _chain(lib, wsb=16) == 1                        # workspace too small
    assert b"workspace too small" in lib.spec_last_error()
    assert _chain(lib, ws=8, wsb=1 << 30) == 1             # misaligned workspace
    assert _chain(lib, B=0) == 0                           # empty batch: nothing to do
    assert lib.spec_adaptive_len(None, 4, 8, ctypes.c_float(0.0), ctypes.c_float(0.1), 1, None, None, 1, 1,
                                 None) == 1                # a must be > 0
    assert lib.spec_tree_build(1, 10, 10, 2, 17, 10, 8, 1, 1, 1, 1, 1, 1, 1, 16, 1 << 30, None) == 2


def test_package_import_is_lazy_and_fails_loudly(tmp_path, monkeypatch):
    # a missing library is an error, never a silent fallback
    monkeypatch.setattr(sv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(sv.SpecError):
        sv.lib()


def test_shape_limits_rejected_on_host(lib):
    # documented shape limits are refused before any device work
    assert _chain(lib, K=4097) == 2
    assert b"K > 4096" in lib.spec_last_error()
    assert lib.spec_verify_greedy(1, 0, 0, 10, 1, 2, 4097, 10, None, None, 1, 1, 1, 16, 1 << 30, None) == 2
    assert lib.spec_verify_tree(1, 0, 0, 10, 1, 1, 1, 2, 8193, 10, 4, 1, 1, 1, 1, 16, 1 << 30, None) == 2
    assert b"N > 8192" in lib.spec_last_error()
    assert lib.spec_tree_build(1, 10, 10, 2, 4, 10, 257, 1, 1, 1, 1, 1, 1, 1, 16, 1 << 30, None) == 2


def test_binding_refuses_unpinned_host_tensors(lib):
    """Host tensors reach the kernels only when pinned (read in place through
    the device mapping); an ordinary host tensor is refused before the call."""
    import torch
    t = torch.zeros(1, 1, 8)
    with pytest.raises(sv.SpecError, match="pinned host tensor"):
        sv.verify_chain(t, torch.zeros(1, 0, 8), torch.zeros(1, 0, dtype=torch.int32), torch.zeros(1, 1), 1.0, 0)
    with pytest.raises(sv.SpecError, match="pinned host tensor"):
        sv.tree_build(torch.zeros(1, 2, 8), 4)
