"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from score_top_expert_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    import score_top_expert_gb300.router as r
    return r.lib()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"MR_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_router_calls():
    names = declared_functions()
    for n in ("router_topk_fwd", "router_topk_bwd", "router_aux_scores_fwd",
              "router_aux_scores_bwd", "moe_router_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(L, n)


def test_library_is_built_for_sm_103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)
    assert B.up_to_date()


def test_version_and_strerror(L):
    assert L.moe_router_version() == 100
    for code in (0, -1, -2, -3, 12345):
        assert isinstance(L.moe_router_strerror(code), bytes)
    assert L.moe_router_strerror(-1) == b"invalid argument"


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails its checks


def fwd(L, **kw):
    a = dict(logits=FAKE, dtype=0, T=4, E=16, K=2, sf=0, ng=0, gk=0, c=1.0, bias=None,
             probs=FAKE, rmap=FAKE, scores=FAKE)
    a.update(kw)
    return L.router_topk_fwd(a["logits"], a["dtype"], a["T"], a["E"], a["K"], a["sf"],
                             a["ng"], a["gk"], a["c"], a["bias"], a["probs"], a["rmap"],
                             a["scores"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), -1), (dict(E=0), -1), (dict(K=0), -1), (dict(K=17), -1),
    (dict(dtype=2), -1), (dict(sf=3), -1), (dict(T=1 << 20, E=4096, K=4), -1),
    (dict(logits=None), -1), (dict(probs=None), -1), (dict(rmap=None), -1),
    (dict(scores=None), -1), (dict(ng=-1), -1),
    (dict(ng=3, gk=1), -1),                   # E % num_groups != 0
    (dict(ng=4, gk=0), -1), (dict(ng=4, gk=5), -1),
    (dict(ng=4, gk=2, K=3), -1),              # K % group_topk != 0
    (dict(ng=4, gk=1, K=8), -1),              # K / group_topk > E / num_groups
    (dict(E=2305, K=4), -2), (dict(E=2304, K=37), -2),
    (dict(E=64, K=4, ng=64, gk=4), -2),       # more groups than supported
])
def test_topk_fwd_rejects(L, kw, code):
    assert fwd(L, **kw) == code


def test_topk_fwd_zero_tokens_is_a_noop(L):
    # T = 0 passes the checks and returns without launching anything
    assert fwd(L, T=0, logits=None) == 0
    assert fwd(L, T=0, logits=None, probs=None, rmap=None, scores=None) == 0
    assert fwd(L, T=0, logits=None, ng=4, gk=2, K=4) == 0


def test_other_calls_reject(L):
    f = FAKE
    assert L.router_topk_bwd(None, f, f, 0, 4, 16, 2, 0, 1.0, f, None) == -1
    assert L.router_topk_bwd(f, f, f, 0, 4, 16, 2, 0, 1.0, None, None) == -1
    assert L.router_topk_bwd(None, None, None, 0, 0, 16, 2, 0, 1.0, None, None) == 0
    assert L.router_topk_bwd(f, f, f, 0, 4, 16, 17, 0, 1.0, f, None) == -1
    assert L.router_topk_bwd(f, f, f, 0, 4, 4000, 2, 0, 1.0, f, None) == -2
    assert L.router_topk_bwd(None, None, None, 0, 0, 16, 2, 0, 1.0, f, None) == 0
    # sigmoid aux needs the intermediate; softmax does not
    assert L.router_aux_scores_fwd(f, 0, 4, 16, 2, 1, f, f, None, None) == -1
    assert L.router_aux_scores_fwd(f, 0, 4, 16, 2, 0, None, f, None, None) == -1
    assert L.router_aux_scores_fwd(None, 0, 0, 16, 2, 0, f, f, None, None) == 0
    assert L.router_aux_scores_bwd(None, f, 0, 4, 16, 2, 0, f, None) == -1
    assert L.router_aux_scores_bwd(f, f, 1, 4, 16, 0, 0, f, None) == -1
    assert L.router_aux_scores_bwd(None, None, 1, 0, 16, 2, 1, f, None) == 0
    # the aux scores take softmax or sigmoid only (not the post-softmax)
    assert L.router_aux_scores_fwd(f, 0, 4, 16, 2, 2, f, f, f, None) == -1
    assert L.router_aux_scores_bwd(f, f, 0, 4, 16, 2, 2, f, None) == -1


def test_path_knobs(L):
    assert L.moe_router_force_path(7) == -1
    prev = L.moe_router_force_path(1)
    assert prev in (0, 1, 2)
    assert L.moe_router_force_path(prev) == 1
    assert L.moe_router_force_fwd_lanes(12) == -1
    p = L.moe_router_force_fwd_lanes(16)
    assert L.moe_router_force_fwd_lanes(p) == 16


def test_product_path_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import score_top_expert_gb300.router as r
    monkeypatch.setattr(r, "_lib", None)
    monkeypatch.setattr(r._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        r.lib()


def test_selftest_rejects_out_of_range_timeouts(L):
    assert L.moe_router_selftest_bounded_wait(0, None) == -1
    assert L.moe_router_selftest_bounded_wait(1000001, None) == -1


def test_aux_loss_argument_checks(L):
    L.router_aux_loss_workspace_bytes.restype = ctypes.c_size_t
    assert L.router_aux_loss_workspace_bytes(8192, 2304) == 64 * 2304 * 8 + 1040
    assert L.router_aux_loss_workspace_bytes(10, 64) == 10 * 64 * 8 + 1040
    assert L.router_aux_loss_workspace_bytes(0, 64) == 0
    f, c = FAKE, ctypes.c_float(0.01)
    big = ctypes.c_size_t(1 << 30)
    fwd = L.router_aux_loss_fwd
    assert fwd(f, f, 4, 16, 17, c, f, f, f, big, None) == -1          # K > E
    assert fwd(f, f, -1, 16, 2, c, f, f, f, big, None) == -1
    assert fwd(f, f, 4, 4000, 2, c, f, f, f, big, None) == -2
    assert fwd(f, f, 4, 16, 2, c, None, f, f, big, None) == -1        # no loss output
    assert fwd(f, f, 4, 16, 2, c, f, f, f, ctypes.c_size_t(16), None) == -1  # workspace too small
    assert fwd(f, f, 4, 16, 2, c, f, f, ctypes.c_void_p(0x1001), big, None) == -1  # misaligned
    assert fwd(None, None, 0, 16, 2, c, None, None, None, ctypes.c_size_t(0), None) == 0
    bwd = L.router_aux_loss_bwd
    assert bwd(f, None, 4, 16, 2, c, f, None) == -1
    assert bwd(None, None, 0, 16, 2, c, None, None) == 0


def test_aux_loss_noalloc_argument_checks(L):
    f, c = FAKE, ctypes.c_float(0.01)
    fwd = L.router_aux_loss_fwd_noalloc
    assert fwd(f, f, 4, 2305, 2, c, f, f, None) == -2    # beyond the scratch array
    assert fwd(f, f, 4, 16, 17, c, f, f, None) == -1
    assert fwd(f, f, 4, 16, 2, c, None, f, None) == -1
    assert fwd(None, None, 0, 16, 2, c, None, None, None) == 0


def test_topk_fwd_compact_rejects(L):
    f, c = FAKE, 1.0
    fn = L.router_topk_fwd_compact
    # (logits, dtype, T, E, K, sf, ng, gk, c, bias, w, ldw, idx, ldi, tei, probs, map, scores)
    assert fn(f, 0, 4, 16, 2, 0, 0, 0, c, None, f, 1, f, 2, None, None, None, None, None) == -1
    assert fn(f, 0, 4, 16, 2, 0, 0, 0, c, None, f, 2, f, 1, None, None, None, None, None) == -1
    assert fn(f, 0, 4, 16, 2, 0, 0, 0, c, None, None, 2, f, 2, None, None, None, None, None) == -1
    assert fn(f, 0, 4, 16, 2, 0, 0, 0, c, None, f, 2, None, 2, None, None, None, None, None) == -1
    assert fn(None, 0, 4, 16, 2, 0, 0, 0, c, None, f, 2, f, 2, None, None, None, None, None) == -1
    assert fn(f, 0, 4, 16, 17, 0, 0, 0, c, None, f, 17, f, 17, None, None, None, None, None) == -1
    assert fn(f, 0, 4, 2305, 2, 0, 0, 0, c, None, f, 2, f, 2, None, None, None, None, None) == -2
    assert fn(f, 0, 4, 16, 3, 0, 4, 2, c, None, f, 3, f, 3, None, None, None, None, None) == -1
    assert fn(None, 0, 0, 16, 2, 0, 0, 0, c, None, None, 2, None, 2, None, None, None, None,
              None) == 0


def test_expert_maps_rejects(L):
    f, big = FAKE, ctypes.c_size_t(1 << 30)
    L.router_expert_maps_workspace_bytes.restype = ctypes.c_size_t
    assert L.router_expert_maps_workspace_bytes(8192, 2304) == (128 + 1) * 2304 * 4 + 16
    assert L.router_expert_maps_workspace_bytes(0, 64) == 0
    fn = L.router_expert_maps
    assert fn(f, 4, 10, 64, 8, f, f, f, f, f, big, None) == -1        # ld < K
    assert fn(f, 8, 10, 64, 65, f, f, f, f, f, big, None) == -1       # K > E
    assert fn(f, 8, 10, 4000, 8, f, f, f, f, f, big, None) == -2
    assert fn(f, 8, 10, 64, 8, f, None, f, f, f, big, None) == -1
    assert fn(f, 8, 10, 64, 8, f, f, f, f, f, ctypes.c_size_t(64), None) == -1
    assert fn(f, 8, 10, 64, 8, f, f, f, f, ctypes.c_void_p(0x1008), big, None) == -1
    assert fn(None, 8, 0, 64, 8, None, None, None, None, None, ctypes.c_size_t(0), None) == 0
    m = L.router_topk_fwd_maps
    # (logits, dt, T, E, K, sf, ng, gk, c, bias, w, ldw, idx, ldi, tei, off, p2u, u2p, pexp, ws, wsb)
    assert m(f, 0, 4, 64, 8, 0, 0, 0, 1.0, None, f, 8, f, 8, None, None, f, f, f, None,
             ctypes.c_size_t(0), None) == -1                          # no offsets
    assert m(f, 0, 40, 63, 8, 0, 0, 0, 1.0, None, f, 8, f, 8, None, f, f, f, f, None,
             ctypes.c_size_t(0), None) == -1                          # composed path, no workspace
    assert m(f, 0, 4, 64, 8, 0, 0, 0, 1.0, None, f, 7, f, 8, None, f, f, f, f, None,
             ctypes.c_size_t(0), None) == -1
    assert m(None, 0, 0, 64, 8, 0, 0, 0, 1.0, None, None, 8, None, 8, None, None, None, None,
             None, None, ctypes.c_size_t(0), None) == 0


def test_cpython_shim_returns_the_c_status_codes():
    # the CPython entry points of the hot calls convert their arguments and
    # return the library's status, exactly as the ctypes entry points do
    import os

    import score_top_expert_gb300.router as R
    from score_top_expert_gb300 import build as B
    if not os.path.exists(B.PYCALLS):
        pytest.skip("interpreter headers absent: the shim is not built")
    L = R.lib()
    fast = R._calls()
    assert not isinstance(fast, R._CtypesCalls)
    cases = [
        ("router_topk_fwd", (0, 0, 0, 64, 4, 0, 0, 0, 1.0, 0, 0, 0, 0, 0)),   # T = 0
        ("router_topk_fwd", (0, 0, 1, 4, 8, 0, 0, 0, 1.0, 0, 0, 0, 0, 0)),    # K > E
        ("router_topk_fwd", (8, 0, 1, 4096, 8, 0, 0, 0, 1.0, 0, 8, 8, 8, 0)),  # E > 2304
        ("router_topk_fwd", (8, 3, 1, 64, 4, 0, 0, 0, 1.0, 0, 8, 8, 8, 0)),   # bad dtype
        ("router_topk_fwd", (8, 0, 1, 64, 4, 0, 3, 1, 1.0, 0, 8, 8, 8, 0)),   # E % groups
        ("router_topk_bwd", (0, 0, 0, 0, 0, 64, 4, 0, 1.0, 0, 0)),            # T = 0
        ("router_topk_bwd", (8, 8, 8, 0, 1, 64, 65, 0, 1.0, 8, 0)),           # K > E
        ("router_aux_scores_fwd", (8, 0, 1, 64, 4, 2, 8, 8, 0, 0)),           # post-softmax
        ("router_aux_scores_fwd", (8, 0, 1, 64, 4, 1, 8, 8, 0, 0)),           # sigmoid, no saved
        ("router_aux_scores_bwd", (0, 0, 0, 0, 64, 4, 0, 0, 0)),              # T = 0
        ("router_aux_scores_bwd", (8, 8, 0, 1, 3000, 4, 0, 8, 0)),            # E > 2304
    ]
    for name, args in cases:
        assert getattr(fast, name)(*args) == getattr(L, name)(*args), (name, args)
    with pytest.raises(TypeError):
        fast.router_topk_fwd(0, 0)
    with pytest.raises(OverflowError):
        fast.router_topk_fwd(0, 0, 2 ** 40, 64, 4, 0, 0, 0, 1.0, 0, 0, 0, 0, 0)
