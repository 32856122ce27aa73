"""The C-ABI library loads, exports every symbol include/gdn.h declares, and validates its
arguments on the host (these calls fail before any CUDA work, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdn():
    from gated_delta_rule_07_gb300 import build
    build.build()
    from gated_delta_rule_07_gb300 import gdn as mod
    return mod


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(gdn):
    names = declared_functions()
    assert "gdn_forward" in names and len(names) >= 9
    lib = ctypes.CDLL(gdn.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert set(gdn.EXPORTED) == set(names)


def test_status_strings(gdn):
    for code, name in gdn.STATUS_NAMES.items():
        assert gdn.gdn_status_string(code).startswith(name)
    assert gdn.gdn_status_string(99) == "GDN_UNKNOWN_STATUS"
    assert gdn.gdn_version() >= 100


def prob(gdn, **kw):
    base = dict(T=4096, N=1, hk=16, hv=32, K=128, V=128, P=1)
    base.update(kw)
    return gdn.make_problem(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(), 0), (dict(P=64, T=65536), 0), (dict(N=8, P=4), 0),
    (dict(hk=3), 1), (dict(hv=0), 1), (dict(P=0), 1), (dict(N=0), 1), (dict(T=-1), 1),
    (dict(K=96), 2), (dict(V=256), 2), (dict(chunk=32), 2), (dict(K=64, V=64), 0),
])
def test_check_problem(gdn, kw, status):
    p = prob(gdn, **kw)
    assert gdn.gdn_check_problem(p) == status
    assert (gdn.gdn_workspace_size(p) > 0) == (status == 0)


def test_workspace_size_accounts_for_segments(gdn):
    p1 = prob(gdn, T=65536, P=1)
    p16 = prob(gdn, T=65536, P=16)
    per_seg = 32 * 128 * 128 * 4 * 3  # M, U, h_in
    assert gdn.gdn_workspace_size(p16) - gdn.gdn_workspace_size(p1) >= 16 * per_seg
    simt = prob(gdn, T=65536, P=1, K=64, V=64)
    # the CUDA-core kernels (K = V = 64) materialise w, u and gcum in fp32
    assert gdn.gdn_workspace_size(simt) >= 65536 * 32 * ((64 + 64) * 4 + 4)


def test_entry_points_reject_bad_arguments_before_any_launch(gdn):
    p = prob(gdn)
    fake = 1 << 20  # never dereferenced: validation fails first
    L = gdn._lib
    by = ctypes.byref
    # null required pointers
    assert L.gdn_forward(by(p), None, fake, fake, fake, fake, None, None, fake, None, fake,
                         1 << 40, None) == 1
    # misaligned q
    assert L.gdn_forward(by(p), fake + 2, fake, fake, fake, fake, None, None, fake, None, fake,
                         1 << 40, None) == 1
    # workspace too small / missing
    assert L.gdn_forward(by(p), fake, fake, fake, fake, fake, None, None, fake, None, fake,
                         16, None) == 3
    assert L.gdn_forward(by(p), fake, fake, fake, fake, fake, None, None, fake, None, None,
                         1 << 40, None) == 3
    # several sequences need cu_seqlens
    p8 = prob(gdn, N=8)
    assert L.gdn_forward(by(p8), fake, fake, fake, fake, fake, None, None, fake, None, fake,
                         1 << 40, None) == 1
    # unsupported shape
    assert L.gdn_forward(by(prob(gdn, K=96)), fake, fake, fake, fake, fake, None, None, fake,
                         None, fake, 1 << 40, None) == 2
    assert L.gdn_chunk_prepare(by(p), None, fake, fake, fake, None, fake, fake, fake, None,
                               None) == 1
    assert L.gdn_segment_summary(by(p), fake, fake, fake, fake, None, None, fake, None,
                                 None) == 1
    assert L.gdn_state_prefix_scan(by(p), fake, fake, None, None, None, None) == 1
    assert L.gdn_chunk_emit(by(p), fake, fake, fake, fake, fake, None, None, None, None, None,
                            None) == 1
    assert L.gdn_device_status(None, 0, None) == 1
    assert L.gdn_forward(None, fake, fake, fake, fake, fake, None, None, fake, None, fake,
                         1 << 40, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The binding refuses to import when libgdn.so is absent (no silent fallback)."""
    import importlib
    import sys
    from gated_delta_rule_07_gb300 import build
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    saved = sys.modules.pop("gated_delta_rule_07_gb300.gdn", None)
    try:
        with pytest.raises(ImportError):
            importlib.import_module("gated_delta_rule_07_gb300.gdn")
    finally:
        sys.modules.pop("gated_delta_rule_07_gb300.gdn", None)
        if saved is not None:
            sys.modules["gated_delta_rule_07_gb300.gdn"] = saved


def test_forward_with_limits_rejects_bad_limits_on_the_host(gdn):
    """A negative wait limit or an unknown fault is rejected before any device work."""
    p = prob(gdn, T=64)
    fake = 1 << 20
    for wc, fault in ((-1, 0), (0, 2), (0, -1)):
        rc = gdn._lib.gdn_forward_with_limits(gdn.ctypes.byref(p), fake, fake, fake, fake, fake,
                                              None, None, fake, None, fake, 1 << 30, None, wc,
                                              fault)
        assert rc == 1


@pytest.mark.parametrize("kw,status", [
    (dict(), 0), (dict(B=0), 0), (dict(K=64, V=64), 0), (dict(K=128, V=64), 0),
    (dict(B=-1), 1), (dict(slots=0), 1), (dict(hk=3), 1), (dict(hv=0), 1),
    (dict(K=96), 2), (dict(V=32), 2), (dict(dtype=None), 2),
])
def test_check_decode_problem(gdn, kw, status):
    base = dict(B=64, slots=128, hk=16, hv=32, K=128, V=128)
    dtype = kw.pop("dtype", "bf16")
    base.update(kw)
    if dtype is None:  # an io dtype outside gdn_dtype
        p = gdn.DecodeProblem(base["B"], base["slots"], base["hk"], base["hv"], base["K"],
                              base["V"], 9)
    else:
        p = gdn.make_decode_problem(**base)
    assert gdn.gdn_check_decode_problem(p) == status


def test_decode_step_rejects_bad_arguments_before_any_launch(gdn):
    p = gdn.make_decode_problem(8, 16, 16, 32, 128, 128)
    fake = 1 << 20
    L = gdn._lib
    by = ctypes.byref
    # null slot table, null state, misaligned q, bad problem
    assert L.gdn_decode_step(by(p), fake, fake, fake, fake, fake, None, fake, fake, None,
                             None) == 1
    assert L.gdn_decode_step(by(p), fake, fake, fake, fake, fake, fake, None, fake, None,
                             None) == 1
    assert L.gdn_decode_step(by(p), fake + 4, fake, fake, fake, fake, fake, fake, fake, None,
                             None) == 1
    assert L.gdn_decode_step(None, fake, fake, fake, fake, fake, fake, fake, fake, None,
                             None) == 1
    # an empty batch is a no-op, whatever the pointers
    p0 = gdn.make_decode_problem(0, 16, 16, 32, 128, 128)
    assert L.gdn_decode_step(by(p0), None, None, None, None, None, None, None, None, None,
                             None) == 0


def test_backward_rejects_bad_arguments_before_any_launch(gdn):
    p = prob(gdn)
    fake = 1 << 20
    L = gdn._lib
    by = ctypes.byref
    args = [fake] * 5 + [None, None, fake, None] + [fake] * 5 + [None]
    # complete call shape: p, q k v g beta, h0, cu, dout, dh_final, dq dk dv dg dbeta, dh0, ws, bytes
    ok = [by(p)] + args[:5] + [None, None, fake, None, fake, fake, fake, fake, fake, None]
    assert L.gdn_backward(*ok, fake, 1, None) == 3           # workspace too small
    bad = list(ok)
    bad[8] = None                                            # no dout
    assert L.gdn_backward(*bad, fake, 1 << 40, None) == 1
    bad = list(ok)
    bad[1] = fake + 8                                        # misaligned q
    assert L.gdn_backward(*bad, fake, 1 << 40, None) == 1
    assert gdn.gdn_backward_workspace_size(prob(gdn, K=96)) == 0
    # the state and state-gradient checkpoints: 2 * 4 * K * V bytes per chunk and value head
    ws = gdn.gdn_backward_workspace_size(prob(gdn, T=65536))
    assert ws >= 2 * (65536 // 64) * 32 * 128 * 128 * 4


def test_prologue_rejects_bad_arguments_before_any_launch(gdn):
    fake = 1 << 20
    L = gdn._lib
    by = ctypes.byref

    def call(**kw):
        base = dict(T=64, N=1, hk=2, hv=4, K=64, V=64, W=4, act=0, io=0)
        base.update(kw)
        p = gdn.PrologueProblem(base["T"], base["N"], base["hk"], base["hv"], base["K"],
                                base["V"], base["W"], base["act"], base["io"])
        return L.gdn_prologue(by(p), fake, fake, None, fake, fake, fake, fake, None, fake, fake,
                              fake, fake, fake, None, None, None)

    assert call(W=5) == 2 and call(W=0) == 2 and call(act=2) == 2 and call(K=256) == 2
    assert call(K=60) == 2 and call(V=12) == 2
    assert call(hk=3) == 1 and call(N=2) == 1 and call(T=-1) == 1 and call(io=5) == 2
    assert L.gdn_prologue(None, fake, fake, None, fake, fake, fake, fake, None, fake, fake, fake,
                          fake, fake, None, None, None) == 1
