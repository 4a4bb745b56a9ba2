"""C ABI checks that need no GPU: the library loads, exports every symbol that
include/dualkv.h declares, and rejects bad arguments with the documented
status codes before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("dualkv.h", "dualkv_layer.h")]


@pytest.fixture(scope="module")
def D():
    from shared_prompt_exact_dualkv_gb300 import build
    if not os.path.exists(build.LIB_PATH):
        build.build()
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv


def declared_functions():
    names = []
    for h in HEADERS:
        names += re.findall(r"DUALKV_API\s+[\w\s\*]+?\b(dualkv_\w+)\s*\(", open(h).read())
    return names


def test_header_declares_expected_entry_points():
    names = set(declared_functions())
    assert {"dualkv_fwd", "dualkv_bwd", "dualkv_bwd_workspace_bytes", "dualkv_status_string",
            "dualkv_last_device_error"} <= names


def test_library_exports_every_declared_symbol(D):
    for name in declared_functions():
        assert hasattr(D.lib, name), name
    assert set(declared_functions()) == set(D.EXPORTED)


def test_status_strings(D):
    for code in range(0, 8):
        assert isinstance(D.dualkv_status_string(code), str) and D.dualkv_status_string(code)
    assert D.dualkv_version() >= 100


def _lens(*r):
    return (ctypes.c_int32 * len(r))(*r)


A = 1 << 20  # a 16-byte aligned fake device address; never dereferenced on these paths


def fwd(D, **kw):
    args = dict(q=A, k=A, v=A, P=128, N=2, R=_lens(64, 64), Hq=2, Hkv=1, d=64, scale=0.125, out=A, lse=A)
    args.update(kw)
    return D.lib.dualkv_fwd(args["q"], args["k"], args["v"], args["P"], args["N"], args["R"], args["Hq"],
                            args["Hkv"], args["d"], args["scale"], args["out"], args["lse"], None)


def bwd(D, **kw):
    args = dict(q=A, k=A, v=A, out=A, dout=A, lse=A, P=128, N=2, R=_lens(64, 64), Hq=2, Hkv=1, d=64,
                scale=0.125, det=0, splits=0, ws=A, ws_bytes=1 << 30, dq=A, dk=A, dv=A)
    args.update(kw)
    return D.lib.dualkv_bwd(args["q"], args["k"], args["v"], args["out"], args["dout"], args["lse"], args["P"],
                            args["N"], args["R"], args["Hq"], args["Hkv"], args["d"], args["scale"], args["det"],
                            args["splits"], args["ws"], args["ws_bytes"], args["dq"], args["dk"], args["dv"], None)


def test_fwd_argument_errors(D):
    assert fwd(D, N=0) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, N=1025) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, R=None) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, P=-1) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, R=_lens(64, -1)) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, d=96) == D.DUALKV_ERR_UNSUPPORTED
    assert fwd(D, Hq=3, Hkv=2) == D.DUALKV_ERR_UNSUPPORTED
    assert fwd(D, Hq=4097, Hkv=1) == D.DUALKV_ERR_UNSUPPORTED   # a grid of items x heads stays in launch limits
    assert fwd(D, Hkv=0) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, q=None) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, lse=None) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(D, k=A + 8) == D.DUALKV_ERR_ALIGNMENT
    assert fwd(D, out=A + 2) == D.DUALKV_ERR_ALIGNMENT
    assert fwd(D, scale=float("nan")) == D.DUALKV_ERR_INVALID_ARG
    # a prompt or response of more than 65535 tiles of 128 rows
    assert fwd(D, P=0, N=1, R=_lens(128 * 65535 + 1)) == D.DUALKV_ERR_UNSUPPORTED
    assert fwd(D, P=128 * 65535 + 1) == D.DUALKV_ERR_UNSUPPORTED
    # empty input is a no-op, whatever the pointers
    assert fwd(D, P=0, N=2, R=_lens(0, 0), q=None, out=None) == D.DUALKV_OK


def test_bwd_argument_errors(D):
    assert bwd(D, N=0) == D.DUALKV_ERR_INVALID_ARG
    assert bwd(D, d=32) == D.DUALKV_ERR_UNSUPPORTED
    assert bwd(D, Hq=8192, Hkv=2) == D.DUALKV_ERR_UNSUPPORTED
    assert bwd(D, dout=None) == D.DUALKV_ERR_INVALID_ARG
    assert bwd(D, dq=A + 4) == D.DUALKV_ERR_ALIGNMENT
    assert bwd(D, ws=None) == D.DUALKV_ERR_WORKSPACE
    assert bwd(D, ws_bytes=16) == D.DUALKV_ERR_WORKSPACE
    assert bwd(D, ws=A + 16) == D.DUALKV_ERR_ALIGNMENT
    assert bwd(D, P=0, N=1, R=_lens(0)) == D.DUALKV_OK


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("P,R,Hq,Hkv,d", [(128, (64, 64, 64, 64), 2, 1, 64), (300, (200, 0, 131), 4, 2, 128),
                                          (0, (77,), 2, 2, 128)])
def test_workspace_bytes(D, P, R, Hq, Hkv, d):
    T = P + sum(R)
    slice_ = P * Hkv * d * 4
    atomic = D.dualkv_bwd_workspace_bytes(P, R, Hq, Hkv, d, False, 0)
    assert atomic == _align256(T * Hq * 4) + 2 * _align256(slice_)
    # the fused-dQ mode adds the fp32 dQ accumulator [Hq][d/4][T][4]
    fused = D.dualkv_bwd_workspace_bytes(P, R, Hq, Hkv, d, 2, 0)
    assert fused == _align256(T * Hq * 4) + 2 * _align256(slice_) + _align256(T * Hq * d * 4)
    assert D.dualkv_bwd_workspace_bytes(P, R, Hq, Hkv, d, 3, 0) == 0
    for S in (1, 2, 3):
        det = D.dualkv_bwd_workspace_bytes(P, R, Hq, Hkv, d, True, S)
        S_eff = max(1, min(S, len(R)))
        assert det == _align256(T * Hq * 4) + 2 * _align256(S_eff * slice_)
    assert D.dualkv_bwd_workspace_bytes(P, R, Hq, Hkv, 96, False, 0) == 0


def test_trace_api_on_cpu(D):
    D.dualkv_trace_enable(True)
    assert all(v == (0.0, 0) for v in D.dualkv_trace_read().values())
    D.dualkv_trace_enable(False)
    assert D.lib.dualkv_trace_read(None, None, 5) == D.DUALKV_ERR_INVALID_ARG


def _grp(D, groups):
    return D._groups(groups)


def fwd_groups(D, groups=((128, (64, 64)), (0, (5,))), G=None, P=None, N=None, R=None, **kw):
    g, Ps, Ns, Rs = _grp(D, groups)
    args = dict(q=A, k=A, v=A, Hq=2, Hkv=1, d=64, scale=0.125, out=A, lse=A)
    args.update(kw)
    return D.lib.dualkv_fwd_groups(args["q"], args["k"], args["v"], g if G is None else G, Ps if P is None else P,
                                   Ns if N is None else N, Rs if R is None else R, args["Hq"], args["Hkv"],
                                   args["d"], args["scale"], args["out"], args["lse"], None)


def test_fwd_groups_argument_errors(D):
    assert fwd_groups(D, G=0) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_groups(D, groups=((-1, (4,)),)) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_groups(D, groups=((4, (4, -2)),)) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_groups(D, N=(ctypes.c_int32 * 2)(2, -1)) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_groups(D, P=ctypes.cast(None, ctypes.POINTER(ctypes.c_int64))) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_groups(D, R=ctypes.cast(None, ctypes.POINTER(ctypes.c_int32))) == D.DUALKV_ERR_INVALID_ARG
    # at most 1040 segments (groups + responses) per call
    ws = D.dualkv_bwd_groups_workspace_bytes
    assert ws([(1, (1,) * 519), (1, (1,) * 519)], 2, 1, 64, False, 0) > 0
    assert ws([(1, (1,) * 519), (1, (1,) * 520)], 2, 1, 64, False, 0) == 0
    assert ws([(1, (1,) * 1039)], 2, 1, 64, False, 0) > 0
    assert fwd_groups(D, groups=[(1, (1,) * 1040)]) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_groups(D, d=96) == D.DUALKV_ERR_UNSUPPORTED
    assert fwd_groups(D, groups=((128 * 65535 + 1, ()),)) == D.DUALKV_ERR_UNSUPPORTED
    assert fwd_groups(D, out=A + 2) == D.DUALKV_ERR_ALIGNMENT
    # groups without responses need no R array; all-empty groups are a no-op
    assert fwd_groups(D, groups=((0, ()), (0, (0, 0))), q=None) == D.DUALKV_OK
    assert fwd_groups(D, groups=((0, ()),), R=ctypes.cast(None, ctypes.POINTER(ctypes.c_int32)),
                      q=None) == D.DUALKV_OK


@pytest.mark.parametrize("groups,Hq,Hkv,d", [(((128, (64, 64)), (0, (5,)), (300, ())), 2, 1, 64),
                                             (((33, (7,)), (0, (9, 9)), (100, (1, 2, 3))), 4, 2, 128)])
def test_groups_workspace_bytes(D, groups, Hq, Hkv, d):
    T = sum(p + sum(r) for p, r in groups)
    slice_ = sum(p for p, _ in groups) * Hkv * d * 4
    atomic = D.dualkv_bwd_groups_workspace_bytes(groups, Hq, Hkv, d, False, 0)
    assert atomic == _align256(T * Hq * 4) + 2 * _align256(slice_)
    assert (D.dualkv_bwd_groups_workspace_bytes(groups, Hq, Hkv, d, 2, 0) ==
            _align256(T * Hq * 4) + 2 * _align256(slice_) + _align256(T * Hq * d * 4))
    maxN = max(len(r) for _, r in groups)
    for S in (1, 2, 3):
        det = D.dualkv_bwd_groups_workspace_bytes(groups, Hq, Hkv, d, True, S)
        assert det == _align256(T * Hq * 4) + 2 * _align256(max(1, min(S, maxN)) * slice_)


@pytest.mark.parametrize("P,R,Hq,Hkv,d", [(128, (64, 64, 64, 64), 2, 1, 64), (300, (200, 0, 131), 4, 2, 128)])
def test_one_group_workspace_matches_single_prompt_call(D, P, R, Hq, Hkv, d):
    for det in (0, 1, 2):
        for S in (0, 1, 2):
            assert (D.dualkv_bwd_groups_workspace_bytes([(P, R)], Hq, Hkv, d, det, S) ==
                    D.dualkv_bwd_workspace_bytes(P, R, Hq, Hkv, d, det, S))


# --------------------------------------------------------------------------- packed decoder layer

def test_packed_positions_match_oracle(D):
    from oracle import layer as L
    groups = [(5, (3, 0, 4)), (0, (2, 6)), (7, ()), (2, (1,))]
    assert D.dualkv_packed_positions(groups) == list(L.packed_positions(groups))


def test_layer_argument_errors(D):
    cfg = D.layer_config(256, 4, 2, 64, 512)
    groups = [(128, (64, 64))]
    assert D.dualkv_layer_workspace_bytes(cfg, groups) > 0
    for bad, code in ((D.layer_config(256, 4, 2, 96, 512), 0), (D.layer_config(252, 4, 2, 64, 512), 0),
                      (D.layer_config(256, 3, 2, 64, 512), 0), (D.layer_config(256, 4, 2, 64, 512, eps=-1.0), 0),
                      (D.layer_config(256, 4, 2, 64, 512, rope_base=0.5), 0),
                      (D.layer_config(256, 8192, 2, 64, 512), 0), (D.layer_config(256, 4, 2, 64, (1 << 24) + 8), 0)):
        assert D.dualkv_layer_workspace_bytes(bad, groups) == code
    assert D.dualkv_layer_workspace_bytes(cfg, [(-1, (4,))]) == 0
    G, Ps, Ns, Rs = D._groups(groups)
    W = D.LayerWeights(*([A] * 6))
    gr = D.LayerGrads(*([A] * 6))
    ws = D.dualkv_layer_workspace_bytes(cfg, groups)
    fwd = lambda **kw: D.lib.dualkv_layer_fwd(ctypes.byref(kw.get("cfg", cfg)), ctypes.byref(kw.get("W", W)),
                                               kw.get("x", A), G, Ps, Ns, Rs, kw.get("y", A), kw.get("ws", A),
                                               kw.get("nbytes", ws), None)
    assert fwd(cfg=D.layer_config(256, 4, 2, 96, 512)) == D.DUALKV_ERR_UNSUPPORTED
    assert fwd(W=D.LayerWeights(*([A] * 5 + [None]))) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(W=D.LayerWeights(*([A] * 5 + [A + 8]))) == D.DUALKV_ERR_ALIGNMENT
    assert fwd(x=None) == D.DUALKV_ERR_INVALID_ARG
    assert fwd(ws=A + 16) == D.DUALKV_ERR_ALIGNMENT
    assert fwd(nbytes=ws - 1) == D.DUALKV_ERR_WORKSPACE
    bwd = lambda **kw: D.lib.dualkv_layer_bwd(ctypes.byref(cfg), ctypes.byref(W), A, A, G, Ps, Ns, Rs, A,
                                               ctypes.byref(kw.get("gr", gr)), A, kw.get("nbytes", ws), None)
    assert bwd(gr=D.LayerGrads(*([A] * 5 + [None]))) == D.DUALKV_ERR_INVALID_ARG
    assert bwd(nbytes=16) == D.DUALKV_ERR_WORKSPACE


def test_selftest_argument_errors(D):
    assert D.lib.dualkv_selftest_wait_timeout(0, 5, None) == D.DUALKV_ERR_INVALID_ARG
    assert D.lib.dualkv_selftest_wait_timeout(20_000_000_000, 5, None) == D.DUALKV_ERR_INVALID_ARG
    assert D.lib.dualkv_selftest_wait_timeout(1000, 0, None) == D.DUALKV_ERR_INVALID_ARG
    assert D.lib.dualkv_selftest_wait_timeout(1000, 1 << 24, None) == D.DUALKV_ERR_INVALID_ARG


def test_static_scratch_limit_matches_header_constant(D):
    """STATIC_SCRATCH_BYTES in the binding is DUALKV_STATIC_SCRATCH_BYTES of the
    header, and the library refuses exactly the shapes whose workspace exceeds
    it (on a machine without a GPU an accepted shape fails later, at the
    device lookup, with another status)."""
    text = open(HEADERS[0]).read()
    m = re.search(r"#define DUALKV_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == D.STATIC_SCRATCH_BYTES
    R = (ctypes.c_int32 * 1)(0)

    def need(P):
        return D.lib.dualkv_bwd_workspace_bytes(P, 1, R, 1, 1, 64, 0, 0)

    lo, hi = 1, 1 << 20
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= D.STATIC_SCRATCH_BYTES else (lo, mid)
    call = lambda P: D.lib.dualkv_bwd_static_workspace(None, None, None, None, None, None, P, 1, R, 1, 1, 64,
                                                       0.125, 0, 0, None, None, None, None)
    assert call(hi) == D.DUALKV_ERR_WORKSPACE
    assert call(lo) != D.DUALKV_ERR_WORKSPACE


def test_partial_entry_points_argument_errors(D):
    """dualkv_fwd_partial / dualkv_bwd_partial refuse a prompt part that is not
    a tile-aligned sub-range of [0, P) before anything is launched."""
    R = _lens(64, 64)

    def fwd_p(lo, hi, **kw):
        a = dict(q=A, P=300, out=A)
        a.update(kw)
        return D.lib.dualkv_fwd_partial(a["q"], A, A, a["P"], 2, R, 2, 1, 64, 0.125, lo, hi, a["out"], A, None)

    def bwd_p(lo, hi, **kw):
        a = dict(dqp=None, dkp=None, dvp=None, ws_bytes=1 << 30)
        a.update(kw)
        return D.lib.dualkv_bwd_partial(A, A, A, A, A, A, 300, 2, R, 2, 1, 64, 0.125, 0, 0, lo, hi, A, a["ws_bytes"],
                                        A, A, A, a["dqp"], a["dkp"], a["dvp"], None)

    for lo, hi in ((64, 128), (0, 200), (128, 0), (-128, 128), (0, 301), (301, 301), (256, 384)):
        assert fwd_p(lo, hi) == D.DUALKV_ERR_INVALID_ARG, (lo, hi)
        assert bwd_p(lo, hi) == D.DUALKV_ERR_INVALID_ARG, (lo, hi)
    assert fwd_p(0, 128, q=None) == D.DUALKV_ERR_INVALID_ARG
    assert fwd_p(0, 128, out=A + 8) == D.DUALKV_ERR_ALIGNMENT
    assert bwd_p(0, 300, dqp=A + 4) == D.DUALKV_ERR_ALIGNMENT
    assert bwd_p(0, 300, dvp=A + 8) == D.DUALKV_ERR_ALIGNMENT
    assert bwd_p(0, 300, ws_bytes=16) == D.DUALKV_ERR_WORKSPACE


def test_checks_build_compiles_and_reports_itself(D):
    """The checks build links with the same exports; only it reports
    dualkv_checks_enabled() == 1 (loaded in a child process)."""
    import subprocess
    import sys
    from shared_prompt_exact_dualkv_gb300 import build
    build.build(checks=True)
    code = ("from shared_prompt_exact_dualkv_gb300 import dualkv as D; "
            "print(D.lib.dualkv_checks_enabled(), all(hasattr(D.lib, n) for n in D.EXPORTED))")
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, DUALKV_LIBRARY="checks"), cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.stdout.split() == ["1", "True"], r.stdout + r.stderr
    assert D.lib.dualkv_checks_enabled() == 0


def test_gemm_argument_errors(D):
    """dualkv_gemm rejects bad arguments before anything touches the GPU."""
    g = lambda kind=0, M=64, N=64, K=64, a=A, b=A, y=A: D.lib.dualkv_gemm(kind, M, N, K, a, b, y, 0, None)
    assert g(kind=3) == D.DUALKV_ERR_INVALID_ARG
    assert g(M=-1) == D.DUALKV_ERR_INVALID_ARG
    assert g(K=1 << 31) == D.DUALKV_ERR_INVALID_ARG
    assert g(N=12) == D.DUALKV_ERR_UNSUPPORTED                  # a row length not a multiple of 8
    assert g(M=(1 << 31) - 8, N=(1 << 20)) == D.DUALKV_ERR_UNSUPPORTED   # M * N over 2^40
    assert g(y=None) == D.DUALKV_ERR_INVALID_ARG
    assert g(a=A + 8) == D.DUALKV_ERR_ALIGNMENT
    assert g(M=0) == D.DUALKV_OK                                # empty output: nothing to do
