"""CPU tests of the C ABI: the library loads, exports what include/gdn.h
declares, and its host-side planner and argument checks behave (no GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from tests import util

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_fwd_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from gated_deltanet_linear_fwd_gb300 import build
        build.build()
    return _lib.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_\w+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = header_functions()
    assert {"gdn_cp_plan", "gdn_chunk_fwd", "gdn_status_string", "gdn_get_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libgdn.so does not export {n}"


def test_status_strings(lib):
    for s in range(8):
        assert lib.gdn_status_string(s)
    assert b"unknown" in lib.gdn_status_string(99)


def plan(lib, T, h_qk=2, h_v=8, B=1, cu=None, mode=3, lam=1.0, w=8, tol=1e-4, sms=152, d=128, dtype=0, rule=1):
    from gated_deltanet_linear_fwd_gb300 import _lib as L
    n_seqs = B if cu is None else len(cu) - 1
    dims = L.gdn_dims(B, T, h_qk, h_v, d, d, n_seqs, 0.0, dtype)
    opts = L.gdn_cp_opts(mode, lam, w, tol, sms, rule)
    out = L.gdn_cp_plan_t()
    arr = None if cu is None else (ctypes.c_int32 * len(cu))(*cu)
    st = lib.gdn_cp_plan(ctypes.byref(dims), arr, ctypes.byref(opts), ctypes.byref(out))
    return st, out


@pytest.mark.parametrize("cu,lam,mode", [
    ([0, 32768], 1.0, 1), ([0, 262144, 327680, 344064, 348160], 1.0, 2),
    ([0, 512], 1.0, 1), ([0, 100, 100, 165, 4000], 0.5, 1), ([0, 64 * 97 + 5], 2.25, 2),
    ([0, 32768], 1.0, 0)])
def test_plan_segments_follow_rule(lib, cu, lam, mode):
    st, p = plan(lib, cu[-1], cu=cu, mode=mode, lam=lam)
    assert st == 0
    q8 = round(lam * 256)
    assert p.lambda_q8 == q8
    segs = [util.segments(cu[n + 1] - cu[n], q8, mode == 0) for n in range(len(cu) - 1)]
    assert p.n_seg_total == sum(len(s) for s in segs)
    assert p.max_seg_chunks == max(b - a for s in segs for (a, b) in s)
    # segments cover each sequence in order, balanced to within one chunk
    for s in segs:
        assert s[0][0] == 0 and all(s[i][1] == s[i + 1][0] for i in range(len(s) - 1))
        lens = [b - a for a, b in s]
        assert max(lens) - min(lens) <= 1


def test_plan_sqrt_model(lib):
    # lambda = 1, N = 512 chunks -> L = round(sqrt(512)) = 23 -> 23 segments
    st, p = plan(lib, 32768, mode=1)
    assert st == 0 and p.n_seg_total == 23 and p.max_seg_chunks == 23


def test_plan_auto_mode(lib):
    st, p = plan(lib, 32768, h_v=8, mode=3, sms=152)
    assert st == 0 and p.mode == 2  # 8 heads < 152 SMs -> warmup-with-exact-fallback CP
    st, p = plan(lib, 4096, B=40, h_v=8, mode=3, sms=152)
    assert st == 0 and p.mode == 0 and p.n_seg_total == 40  # 320 chains fill the GPU -> off


def test_plan_records_the_tolerance_rule(lib):
    for rule in (0, 1):
        st, p = plan(lib, 32768, mode=2, rule=rule, tol=3e-4)
        assert st == 0 and p.tol_rule == rule and abs(p.warmup_tol - 3e-4) < 1e-9


def test_plan_workspace_layout(lib):
    st, p = plan(lib, 32768, h_v=8, mode=1)
    mat = 128 * 128 * 4
    assert p.off_head % 256 == 0 and p.off_seg_bound % 256 == 0
    assert p.off_Sloc - p.off_R == 23 * 8 * mat and p.off_Sstart - p.off_Sloc == 23 * 8 * mat
    # chunk index (n_seqs + 1 int32, 16-byte chunk records) and the chunk warmup exponents,
    # then the chunk records
    assert p.n_chunks_total == 512
    assert p.off_chunk_map == p.off_Sstart + 23 * 8 * mat
    assert p.off_wy % 1024 == 0 and p.off_wy >= p.off_chunk_map + 8 + 512 * 16 + 512 * 8 * 4
    assert p.workspace_bytes == p.off_wy + 512 * 8 * 41472
    st, p0 = plan(lib, 32768, h_v=8, mode=0)
    assert p0.off_R == p0.off_Sloc == p0.off_Sstart == 0  # no context parallelism: no segment states
    assert p0.workspace_bytes == p0.off_wy + 512 * 8 * 41472


@pytest.mark.parametrize("kw,expect", [
    (dict(d=64), 2), (dict(dtype=5), 2), (dict(mode=9), 2), (dict(rule=2), 2), (dict(rule=-1), 2), (dict(h_v=0), 1),
    (dict(cu=[0, 10, 5]), 1), (dict(cu=[1, 10]), 1), (dict(cu=[0, 9]), 1), (dict(B=2, cu=[0, 10]), 1)])
def test_plan_rejects(lib, kw, expect):
    T = kw.get("cu", [0, 10])[-1] if "cu" in kw else 10
    if kw.get("cu") == [0, 9]:
        T = 10  # cu does not end at T
    st, _ = plan(lib, T, **kw)
    assert st == expect


def test_chunk_fwd_rejects_before_device_work(lib):
    from gated_deltanet_linear_fwd_gb300 import _lib as L
    st, p = plan(lib, 128, h_qk=1, h_v=1, mode=0)
    assert st == 0
    dims = L.gdn_dims(1, 128, 1, 1, 128, 128, 1, 0.0, 0)
    A = ctypes.c_void_p(0x100000)  # never dereferenced: every case fails a host check first
    U = ctypes.c_void_p(0x100008)  # not 16-byte aligned
    ws = p.workspace_bytes
    f = lib.gdn_chunk_fwd
    # null plan / dims
    assert f(A, A, A, A, A, None, None, A, None, None, ctypes.byref(p), A, ws, None) == 1
    assert f(A, A, A, A, A, None, None, A, None, ctypes.byref(dims), None, A, ws, None) == 1
    # workspace missing or too small
    assert f(A, A, A, A, A, None, None, A, None, ctypes.byref(dims), ctypes.byref(p), None, ws, None) == 6
    assert f(A, A, A, A, A, None, None, A, None, ctypes.byref(dims), ctypes.byref(p), A, 16, None) == 6
    # misaligned
    assert f(U, A, A, A, A, None, None, A, None, ctypes.byref(dims), ctypes.byref(p), A, ws, None) == 3
    assert f(A, A, A, A, A, None, None, A, None, ctypes.byref(dims), ctypes.byref(p), U, ws, None) == 3
    # null input
    assert f(None, A, A, A, A, None, None, A, None, ctypes.byref(dims), ctypes.byref(p), A, ws, None) == 1
    # dims disagree with the plan
    dims2 = L.gdn_dims(1, 128, 1, 2, 128, 128, 1, 0.0, 0)
    assert f(A, A, A, A, A, None, None, A, None, ctypes.byref(dims2), ctypes.byref(p), A, ws, None) == 1
    # unsupported head dim
    dims3 = L.gdn_dims(1, 128, 1, 1, 64, 128, 1, 0.0, 0)
    assert f(A, A, A, A, A, None, None, A, None, ctypes.byref(dims3), ctypes.byref(p), A, ws, None) == 2


def test_bwd_workspace_layout(lib):
    """The backward's workspace: the forward's (rounded up to 1 KB), then per (chunk,
    value head) A^T (8 KB) and four 32 KB tiles, then a bf16 copy of o."""
    st, p = plan(lib, 32768, h_v=8, mode=3)
    assert st == 0
    n = ctypes.c_size_t(0)
    assert lib.gdn_bwd_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    base = -(-p.workspace_bytes // 1024) * 1024
    o_end = base + 512 * 8 * (8192 + 4 * 32768) + 32768 * 8 * 128 * 2
    assert n.value == -(-o_end // 256) * 256
    assert lib.gdn_bwd_workspace_bytes(None, ctypes.byref(n)) == 1
    st, pf = plan(lib, 32768, h_v=8, mode=3, dtype=1)  # the fp32 path has no backward
    assert st == 0 and lib.gdn_bwd_workspace_bytes(ctypes.byref(pf), ctypes.byref(n)) == 2


def test_chunk_bwd_rejects_before_device_work(lib):
    from gated_deltanet_linear_fwd_gb300 import _lib as L
    st, p = plan(lib, 128, h_qk=1, h_v=1, mode=0)
    assert st == 0
    n = ctypes.c_size_t(0)
    assert lib.gdn_bwd_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    ws = n.value
    dims = L.gdn_dims(1, 128, 1, 1, 128, 128, 1, 0.0, 0)
    A = ctypes.c_void_p(0x100000)  # never dereferenced: every case fails a host check first
    U = ctypes.c_void_p(0x100008)  # not 16-byte aligned
    f = lib.gdn_chunk_bwd
    D, P = ctypes.byref(dims), ctypes.byref(p)

    def call(d_out=A, dq=A, dims_=D, plan_=P, work=A, nbytes=ws, dhT=None):
        return f(A, A, A, A, A, None, None, d_out, dhT, dq, A, A, A, A, None, dims_, plan_, work, nbytes, 0, None)

    assert call(dims_=None) == 1 and call(plan_=None) == 1       # null dims / plan
    assert call(nbytes=ws - 1) == 6 and call(work=None) == 6     # workspace missing or too small
    assert call(d_out=None) == 1 and call(dq=None) == 1          # null upstream gradient / output
    assert call(d_out=U) == 3 and call(dhT=U) == 3               # misaligned
    dims32 = L.gdn_dims(1, 128, 1, 1, 128, 128, 1, 0.0, 1)
    assert call(dims_=ctypes.byref(dims32)) == 2                 # fp32: no backward
    g = lib.gdn_chunk_fwd_train
    assert g(A, A, A, A, A, None, None, A, None, D, None, A, ws, None) == 1
    assert g(A, A, A, A, A, None, None, A, None, D, P, A, ws - 1, None) == 6
    assert g(A, A, A, A, A, None, None, A, None, ctypes.byref(dims32), P, A, ws, None) == 2


def test_decode_step_rejects_before_device_work(lib):
    from gated_deltanet_linear_fwd_gb300 import _lib as L
    A = ctypes.c_void_p(0x100000)  # never dereferenced: every case fails a host check first
    U = ctypes.c_void_p(0x100008)  # not 16-byte aligned
    f = lib.gdn_decode_step
    ok = L.gdn_dims(4, 1, 2, 8, 128, 128, 4, 0.0, 0)
    assert f(A, A, A, A, A, A, A, None, None) == 1                                    # null dims
    assert f(A, A, A, A, A, A, A, ctypes.byref(L.gdn_dims(4, 2, 2, 8, 128, 128, 4, 0.0, 0)), None) == 1  # T != 1
    assert f(A, A, A, A, A, A, A, ctypes.byref(L.gdn_dims(4, 1, 2, 8, 128, 128, 3, 0.0, 0)), None) == 1  # n_seqs != B
    assert f(A, A, A, A, A, None, A, ctypes.byref(ok), None) == 1                     # null state
    assert f(A, A, A, A, A, A, U, ctypes.byref(ok), None) == 3                        # misaligned out
    assert f(A, A, A, A, A, A, A, ctypes.byref(L.gdn_dims(4, 1, 2, 8, 64, 128, 4, 0.0, 0)), None) == 2  # d_k


def test_binding_fails_loudly_without_library(tmp_path):
    from gated_deltanet_linear_fwd_gb300 import _lib as L
    saved = L._lib
    try:
        L._lib = None
        with pytest.raises(RuntimeError, match="libgdn.so not found"):
            L.load(str(tmp_path / "missing.so"))
    finally:
        L._lib = saved


@pytest.mark.parametrize("cu,h_v,sms", [([0, 32768], 8, 152), ([0, 32768], 24, 148),
                                        ([0, 262144, 327680, 344064, 348160], 8, 152), ([0, 512], 4, 152),
                                        ([0, 4096, 20480, 86016, 348160], 8, 152),
                                        ([0, 100000, 100100, 160000], 4, 148)])
def test_plan_automatic_lambda(lib, cu, h_v, sms):
    lens = [cu[n + 1] - cu[n] for n in range(len(cu) - 1)]
    st, p = plan(lib, cu[-1], h_v=h_v, cu=cu, mode=2, lam=0.0, sms=sms)
    assert st == 0
    assert p.lambda_q8 == util.auto_lambda_q8(lens, h_v, sms)
    # the fp32 path: two CTAs per SM, no per-CTA overhead, no combine term
    st, p = plan(lib, cu[-1], h_v=h_v, cu=cu, mode=1, lam=0.0, sms=sms, dtype=1)
    assert st == 0
    assert p.lambda_q8 == util.auto_lambda_q8(lens, h_v, 2 * sms, overhead=0, combine=False)


def test_device_status_decoding():
    """The host's reading of the status word's (code, detail) pairs."""
    from gated_deltanet_linear_fwd_gb300 import describe_device_status
    assert describe_device_status(0, 0) == "ok"
    assert describe_device_status(5, 6) == "timeout: the test hook's stall"
    assert describe_device_status(7, 5).startswith("check failed: a value outside the fp16 range")
    assert describe_device_status(7, 3).endswith("disagree with the plan")
    assert describe_device_status(5, 108) == "timeout: the bounded wait on barrier 8"


def test_debug_stall_hook_is_exported_and_settable(lib):
    assert lib.gdn_debug_stall_ns(0) == 0
    assert lib.gdn_debug_stall_ns(1000) == 0
    assert lib.gdn_debug_stall_ns(0) == 0


def test_head_modes_without_a_device_decision(lib):
    """Plans whose heads take no on-device decision report their modes from the
    plan alone, without touching the workspace (a dummy, never-dereferenced
    pointer here): no context parallelism (off), the fp32 path (exact), and a
    plan in which every sequence is one segment (the plan's mode)."""
    from gated_deltanet_linear_fwd_gb300 import _lib as L
    A = ctypes.c_void_p(0x100000)
    cases = [(dict(mode=0), 0), (dict(mode=1, dtype=1, lam=0.5), 1),
             (dict(mode=1, cu=[0, 60, 120]), 1), (dict(mode=2, cu=[0, 60, 120]), 2)]
    for kw, want in cases:
        cu = kw.pop("cu", None)
        T = cu[-1] if cu else 32768
        st, p = plan(lib, T, h_v=4, cu=cu, **kw)
        assert st == 0
        if cu:
            assert p.n_seg_total == p.n_seqs  # one chunk a sequence: one segment each
        n = p.n_seqs * p.h_v
        modes, bounds = (ctypes.c_int32 * n)(), (ctypes.c_float * n)()
        assert lib.gdn_cp_head_modes(A, ctypes.byref(p), modes, bounds, None) == 0
        assert list(modes) == [want] * n, (kw, list(modes))
        assert all(b == float("-inf") for b in bounds)
