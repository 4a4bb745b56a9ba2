"""Python binding of the C ABI in ``include/dualkv.h`` (argument marshalling only).

Every call goes straight to ``libdualkv.so``; all arithmetic runs in the CUDA
kernels.  There is no fallback: if the library is missing, importing this
module raises.  PyTorch is used only to own device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# DUALKV_LIBRARY=checks loads the checks build (libdualkv_checks.so, made by
# build.build(checks=True)) instead of the regular library.
LIB_PATH = os.path.join(_HERE, "libdualkv_checks.so" if os.environ.get("DUALKV_LIBRARY") == "checks"
                        else "libdualkv.so")

DUALKV_OK = 0
DUALKV_ERR_INVALID_ARG = 1
DUALKV_ERR_UNSUPPORTED = 2
DUALKV_ERR_ALIGNMENT = 3
DUALKV_ERR_WORKSPACE = 4
DUALKV_ERR_CUDA = 5
DUALKV_ERR_TIMEOUT = 6
DUALKV_ERR_CHECK = 7

EXPORTED = ("dualkv_fwd", "dualkv_bwd", "dualkv_bwd_workspace_bytes", "dualkv_status_string",
            "dualkv_last_device_error", "dualkv_trace_enable", "dualkv_trace_read", "dualkv_version",
            "dualkv_bwd_static_workspace", "dualkv_fwd_groups", "dualkv_bwd_groups_workspace_bytes",
            "dualkv_bwd_groups", "dualkv_layer_workspace_bytes", "dualkv_layer_fwd", "dualkv_layer_bwd",
            "dualkv_packed_positions", "dualkv_selftest_wait_timeout", "dualkv_fwd_partial", "dualkv_bwd_partial",
            "dualkv_checks_enabled", "dualkv_gemm", "dualkv_last_cuda_error")

# Size of the library's fixed backward scratch (DUALKV_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 16 << 20

TRACE_KERNELS = ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_prompt_reduce", "bwd_dq")


LAYER_WEIGHTS = ("ln1", "wqkv", "wo", "ln2", "wgu", "wd")


class LayerConfig(ctypes.Structure):
    """dualkv_layer_config."""
    _fields_ = [("hidden", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("rope_base", ctypes.c_float), ("eps", ctypes.c_float)]


class LayerWeights(ctypes.Structure):
    """dualkv_layer_weights: device pointers of the bf16 weights."""
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_WEIGHTS]


class LayerGrads(ctypes.Structure):
    """dualkv_layer_grads: device pointers of the fp32 weight gradients."""
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_WEIGHTS]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                          "(python -m shared_prompt_exact_dualkv_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    c_i64, c_i32, c_p, c_f = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_float
    p_i32 = ctypes.POINTER(ctypes.c_int32)
    lib.dualkv_fwd.argtypes = [c_p, c_p, c_p, c_i64, c_i32, p_i32, c_i32, c_i32, c_i32, c_f, c_p, c_p, c_p]
    lib.dualkv_fwd.restype = ctypes.c_int
    lib.dualkv_bwd_workspace_bytes.argtypes = [c_i64, c_i32, p_i32, c_i32, c_i32, c_i32, ctypes.c_int, c_i32]
    lib.dualkv_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.dualkv_bwd.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i32, p_i32, c_i32, c_i32, c_i32, c_f,
                               ctypes.c_int, c_i32, c_p, ctypes.c_size_t, c_p, c_p, c_p, c_p]
    lib.dualkv_bwd.restype = ctypes.c_int
    lib.dualkv_status_string.argtypes = [ctypes.c_int]
    lib.dualkv_status_string.restype = ctypes.c_char_p
    lib.dualkv_last_cuda_error.argtypes = []
    lib.dualkv_last_cuda_error.restype = c_i32
    lib.dualkv_last_device_error.argtypes = [c_p, p_i32]
    lib.dualkv_last_device_error.restype = ctypes.c_int
    lib.dualkv_trace_enable.argtypes = [ctypes.c_int]
    lib.dualkv_trace_enable.restype = ctypes.c_int
    lib.dualkv_trace_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), c_i32]
    lib.dualkv_trace_read.restype = ctypes.c_int
    lib.dualkv_bwd_static_workspace.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i32, p_i32, c_i32, c_i32,
                                                 c_i32, c_f, ctypes.c_int, c_i32, c_p, c_p, c_p, c_p]
    lib.dualkv_bwd_static_workspace.restype = ctypes.c_int
    p_i64 = ctypes.POINTER(ctypes.c_int64)
    lib.dualkv_fwd_groups.argtypes = [c_p, c_p, c_p, c_i32, p_i64, p_i32, p_i32, c_i32, c_i32, c_i32, c_f, c_p,
                                      c_p, c_p]
    lib.dualkv_fwd_groups.restype = ctypes.c_int
    lib.dualkv_bwd_groups_workspace_bytes.argtypes = [c_i32, p_i64, p_i32, p_i32, c_i32, c_i32, c_i32, ctypes.c_int,
                                                      c_i32]
    lib.dualkv_bwd_groups_workspace_bytes.restype = ctypes.c_size_t
    lib.dualkv_bwd_groups.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, p_i64, p_i32, p_i32, c_i32, c_i32,
                                      c_i32, c_f, ctypes.c_int, c_i32, c_p, ctypes.c_size_t, c_p, c_p, c_p, c_p]
    lib.dualkv_bwd_groups.restype = ctypes.c_int
    p_cfg = ctypes.POINTER(LayerConfig)
    lib.dualkv_layer_workspace_bytes.argtypes = [p_cfg, c_i32, p_i64, p_i32, p_i32]
    lib.dualkv_layer_workspace_bytes.restype = ctypes.c_size_t
    lib.dualkv_layer_fwd.argtypes = [p_cfg, ctypes.POINTER(LayerWeights), c_p, c_i32, p_i64, p_i32, p_i32, c_p, c_p,
                                     ctypes.c_size_t, c_p]
    lib.dualkv_layer_fwd.restype = ctypes.c_int
    lib.dualkv_layer_bwd.argtypes = [p_cfg, ctypes.POINTER(LayerWeights), c_p, c_p, c_i32, p_i64, p_i32, p_i32, c_p,
                                     ctypes.POINTER(LayerGrads), c_p, ctypes.c_size_t, c_p]
    lib.dualkv_layer_bwd.restype = ctypes.c_int
    lib.dualkv_packed_positions.argtypes = [c_i32, p_i64, p_i32, p_i32, p_i32, c_i64]
    lib.dualkv_packed_positions.restype = ctypes.c_int
    lib.dualkv_selftest_wait_timeout.argtypes = [c_i64, c_i32, c_p]
    lib.dualkv_selftest_wait_timeout.restype = ctypes.c_int
    lib.dualkv_fwd_partial.argtypes = [c_p, c_p, c_p, c_i64, c_i32, p_i32, c_i32, c_i32, c_i32, c_f, c_i64, c_i64,
                                       c_p, c_p, c_p]
    lib.dualkv_fwd_partial.restype = ctypes.c_int
    lib.dualkv_bwd_partial.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_i64, c_i32, p_i32, c_i32, c_i32, c_i32, c_f,
                                       ctypes.c_int, c_i32, c_i64, c_i64, c_p, ctypes.c_size_t, c_p, c_p, c_p, c_p,
                                       c_p, c_p, c_p]
    lib.dualkv_bwd_partial.restype = ctypes.c_int
    lib.dualkv_gemm.argtypes = [c_i32, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_i32, c_p]
    lib.dualkv_gemm.restype = ctypes.c_int
    lib.dualkv_checks_enabled.argtypes = []
    lib.dualkv_checks_enabled.restype = ctypes.c_int
    lib.dualkv_version.argtypes = []
    lib.dualkv_version.restype = ctypes.c_int
    return lib


lib = _load()


class DualKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.cuda_error = dualkv_last_cuda_error() if status == DUALKV_ERR_CUDA else 0
        detail = f", CUDA code {self.cuda_error}" if self.cuda_error else ""
        super().__init__(f"{where}: {dualkv_status_string(status)} (status {status}{detail})")


def dualkv_last_cuda_error() -> int:
    """The CUDA code behind this thread's most recent DUALKV_ERR_CUDA (0: none)."""
    return int(lib.dualkv_last_cuda_error())


def dualkv_status_string(status: int) -> str:
    return lib.dualkv_status_string(int(status)).decode()


def _lens(R_lens: Sequence[int]):
    arr = (ctypes.c_int32 * len(R_lens))(*[int(r) for r in R_lens])
    return arr


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


BWD_ATOMIC = 0           # fp32 atomics for prompt dK/dV, separate dQ kernel
BWD_DETERMINISTIC = 1    # fixed-order sums, bitwise reproducible
BWD_ATOMIC_FUSED_DQ = 2  # fp32 atomics, dQ fused into the dK/dV kernel (slower on GB300)


def _mode(deterministic) -> int:
    """The backward mode: False/True map to BWD_ATOMIC/BWD_DETERMINISTIC; an
    int is passed through."""
    if isinstance(deterministic, bool):
        return BWD_DETERMINISTIC if deterministic else BWD_ATOMIC
    return int(deterministic)


def _check(st: int, where: str) -> None:
    if st != DUALKV_OK:
        raise DualKVError(st, where)


def dualkv_fwd(q, k, v, P: int, R_lens: Sequence[int], out, lse, softmax_scale: float,
               stream=None, check: bool = True) -> int:
    """Calls dualkv_fwd on device tensors (q/out [T,Hq,d], k/v [T,Hkv,d] bf16, lse [Hq,T] fp32)."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    st = lib.dualkv_fwd(_ptr(q), _ptr(k), _ptr(v), int(P), len(R_lens), _lens(R_lens), Hq, Hkv, d,
                        float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream))
    if check:
        _check(st, "dualkv_fwd")
    return st


def dualkv_bwd_workspace_bytes(P: int, R_lens: Sequence[int], Hq: int, Hkv: int, d: int,
                               deterministic: bool, num_splits: int = 0) -> int:
    return int(lib.dualkv_bwd_workspace_bytes(int(P), len(R_lens), _lens(R_lens), int(Hq), int(Hkv), int(d),
                                              _mode(deterministic), int(num_splits)))


def dualkv_bwd(q, k, v, out, dout, lse, P: int, R_lens: Sequence[int], softmax_scale: float,
               deterministic: bool, workspace, dq, dk, dv, num_splits: int = 0, stream=None,
               check: bool = True) -> int:
    """Calls dualkv_bwd; `workspace` is a uint8 device tensor of at least
    dualkv_bwd_workspace_bytes(...) bytes."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.dualkv_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), int(P), len(R_lens),
                        _lens(R_lens), Hq, Hkv, d, float(softmax_scale), _mode(deterministic),
                        int(num_splits), _ptr(workspace), ws_bytes, _ptr(dq), _ptr(dk), _ptr(dv),
                        _stream(stream))
    if check:
        _check(st, "dualkv_bwd")
    return st


def dualkv_bwd_static_workspace(q, k, v, out, dout, lse, P: int, R_lens: Sequence[int], softmax_scale: float,
                                deterministic: bool, dq, dk, dv, num_splits: int = 0, stream=None,
                                check: bool = True) -> int:
    """Backward pass that allocates nothing: the library's own fixed 16 MiB
    device scratch replaces the workspace (for callers that cannot allocate
    device memory when they run the backward pass).  Calls that can overlap on
    the GPU share that scratch and must be ordered by the caller."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    st = lib.dualkv_bwd_static_workspace(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), int(P),
                                         len(R_lens), _lens(R_lens), Hq, Hkv, d, float(softmax_scale),
                                         _mode(deterministic), int(num_splits), _ptr(dq), _ptr(dk), _ptr(dv),
                                         _stream(stream))
    if check:
        _check(st, "dualkv_bwd_static_workspace")
    return st


def dualkv_fwd_partial(q, k, v, P: int, R_lens: Sequence[int], prompt_rows, out, lse, softmax_scale: float,
                       stream=None, check: bool = True) -> int:
    """Calls dualkv_fwd_partial: the prompt query rows prompt_rows = (lo, hi)
    and every response row."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    lo, hi = prompt_rows
    st = lib.dualkv_fwd_partial(_ptr(q), _ptr(k), _ptr(v), int(P), len(R_lens), _lens(R_lens), Hq, Hkv, d,
                                float(softmax_scale), int(lo), int(hi), _ptr(out), _ptr(lse), _stream(stream))
    if check:
        _check(st, "dualkv_fwd_partial")
    return st


def dualkv_bwd_partial(q, k, v, out, dout, lse, P: int, R_lens: Sequence[int], prompt_rows, softmax_scale: float,
                       deterministic: bool, workspace, dq, dk, dv, dq_prompt=None, dk_prompt=None, dv_prompt=None,
                       num_splits: int = 0, stream=None, check: bool = True) -> int:
    """Calls dualkv_bwd_partial; dq_prompt [P,Hq,d] and dk_prompt/dv_prompt
    [P,Hkv,d] are optional fp32 device tensors for the unrounded prompt rows."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    lo, hi = prompt_rows
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.dualkv_bwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), int(P), len(R_lens),
                                _lens(R_lens), Hq, Hkv, d, float(softmax_scale), _mode(deterministic),
                                int(num_splits), int(lo), int(hi), _ptr(workspace), ws_bytes, _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(dq_prompt), _ptr(dk_prompt), _ptr(dv_prompt), _stream(stream))
    if check:
        _check(st, "dualkv_bwd_partial")
    return st


def _groups(groups):
    """[(P_g, [R_g,0, ...]), ...] -> (G, P array, N array, concatenated R array)."""
    G = len(groups)
    Ps = (ctypes.c_int64 * max(G, 1))(*[int(p) for p, _ in groups])
    Ns = (ctypes.c_int32 * max(G, 1))(*[len(r) for _, r in groups])
    flat = [int(x) for _, r in groups for x in r]
    Rs = (ctypes.c_int32 * max(len(flat), 1))(*flat)
    return G, Ps, Ns, Rs


def dualkv_fwd_groups(q, k, v, groups, out, lse, softmax_scale: float, stream=None, check: bool = True) -> int:
    """Calls dualkv_fwd_groups; `groups` lists (prompt length, response lengths) per group in row order."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G, Ps, Ns, Rs = _groups(groups)
    st = lib.dualkv_fwd_groups(_ptr(q), _ptr(k), _ptr(v), G, Ps, Ns, Rs, Hq, Hkv, d, float(softmax_scale),
                               _ptr(out), _ptr(lse), _stream(stream))
    if check:
        _check(st, "dualkv_fwd_groups")
    return st


def dualkv_bwd_groups_workspace_bytes(groups, Hq: int, Hkv: int, d: int, deterministic: bool,
                                      num_splits: int = 0) -> int:
    G, Ps, Ns, Rs = _groups(groups)
    return int(lib.dualkv_bwd_groups_workspace_bytes(G, Ps, Ns, Rs, int(Hq), int(Hkv), int(d),
                                                     _mode(deterministic), int(num_splits)))


def dualkv_bwd_groups(q, k, v, out, dout, lse, groups, softmax_scale: float, deterministic: bool, workspace,
                      dq, dk, dv, num_splits: int = 0, stream=None, check: bool = True) -> int:
    """Calls dualkv_bwd_groups (argument meaning as dualkv_bwd, layout as dualkv_fwd_groups)."""
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G, Ps, Ns, Rs = _groups(groups)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.dualkv_bwd_groups(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), G, Ps, Ns, Rs, Hq,
                               Hkv, d, float(softmax_scale), _mode(deterministic), int(num_splits),
                               _ptr(workspace), ws_bytes, _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream))
    if check:
        _check(st, "dualkv_bwd_groups")
    return st


def dualkv_gemm(kind: int, A, B, Y, accumulate: bool = False, stream=None, check: bool = True) -> int:
    """The layer's tensor-core GEMM: kind 0 Y = A.B^T (+ Y), kind 1 Y = A.B,
    kind 2 Y (fp32) = A^T.B; A, B bf16 row-major device tensors."""
    if kind == 0:
        M, K = A.shape
        N = B.shape[0]
    elif kind == 1:
        M, K = A.shape
        N = B.shape[1]
    else:
        K, M = A.shape
        N = B.shape[1]
    st = lib.dualkv_gemm(int(kind), int(M), int(N), int(K), _ptr(A), _ptr(B), _ptr(Y), 1 if accumulate else 0,
                         _stream(stream))
    if check:
        _check(st, "dualkv_gemm")
    return st


def dualkv_last_device_error(stream=None):
    """Synchronises the stream and returns (status, site) of the device error word."""
    site = ctypes.c_int32(0)
    st = lib.dualkv_last_device_error(_stream(stream), ctypes.byref(site))
    return st, site.value


def dualkv_selftest_wait_timeout(limit_ns: int, site: int, stream=None) -> None:
    """Launches the bounded-wait self-test (a wait that nothing completes)."""
    _check(lib.dualkv_selftest_wait_timeout(int(limit_ns), int(site), _stream(stream)),
           "dualkv_selftest_wait_timeout")


def dualkv_trace_enable(on: bool) -> None:
    _check(lib.dualkv_trace_enable(1 if on else 0), "dualkv_trace_enable")


def dualkv_trace_read() -> dict:
    """{kernel name: (total device ms, launches)} since the last enable."""
    n = len(TRACE_KERNELS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(lib.dualkv_trace_read(ms, cnt, n), "dualkv_trace_read")
    return {name: (ms[i], cnt[i]) for i, name in enumerate(TRACE_KERNELS)}


def dualkv_version() -> int:
    return int(lib.dualkv_version())


# --------------------------------------------------------------------------- conveniences

def forward(q, k, v, P: int, R_lens: Sequence[int], softmax_scale: Optional[float] = None, stream=None):
    """Allocates out/lse and runs dualkv_fwd; returns (out, lse)."""
    T, Hq, d = q.shape
    if softmax_scale is None:
        softmax_scale = d ** -0.5
    out = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    dualkv_fwd(q, k, v, P, R_lens, out, lse, softmax_scale, stream)
    return out, lse


def backward(q, k, v, out, dout, lse, P: int, R_lens: Sequence[int], softmax_scale: Optional[float] = None,
             deterministic: bool = False, num_splits: int = 0, stream=None, workspace=None):
    """Allocates dq/dk/dv (and the workspace unless given) and runs dualkv_bwd."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if softmax_scale is None:
        softmax_scale = d ** -0.5
    if workspace is None:
        nbytes = dualkv_bwd_workspace_bytes(P, R_lens, Hq, Hkv, d, deterministic, num_splits)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dualkv_bwd(q, k, v, out, dout, lse, P, R_lens, softmax_scale, deterministic, workspace, dq, dk, dv,
               num_splits=num_splits, stream=stream)
    return dq, dk, dv


def forward_groups(q, k, v, groups, softmax_scale: Optional[float] = None, stream=None):
    """Allocates out/lse and runs dualkv_fwd_groups; returns (out, lse)."""
    T, Hq, d = q.shape
    if softmax_scale is None:
        softmax_scale = d ** -0.5
    out = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    dualkv_fwd_groups(q, k, v, groups, out, lse, softmax_scale, stream)
    return out, lse


def backward_groups(q, k, v, out, dout, lse, groups, softmax_scale: Optional[float] = None,
                    deterministic: bool = False, num_splits: int = 0, stream=None, workspace=None):
    """Allocates dq/dk/dv (and the workspace unless given) and runs dualkv_bwd_groups."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if softmax_scale is None:
        softmax_scale = d ** -0.5
    if workspace is None:
        nbytes = dualkv_bwd_groups_workspace_bytes(groups, Hq, Hkv, d, deterministic, num_splits)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dualkv_bwd_groups(q, k, v, out, dout, lse, groups, softmax_scale, deterministic, workspace, dq, dk, dv,
                      num_splits=num_splits, stream=stream)
    return dq, dk, dv


# --------------------------------------------------------------------------- packed decoder layer

def layer_config(hidden: int, Hq: int, Hkv: int, d: int, inter: int, rope_base: float = 1.0e6,
                 eps: float = 1.0e-6) -> LayerConfig:
    return LayerConfig(int(hidden), int(Hq), int(Hkv), int(d), int(inter), float(rope_base), float(eps))


def layer_weight_shapes(cfg: LayerConfig) -> dict:
    """Shapes of the bf16 weights (and of the fp32 gradients)."""
    return {"ln1": (cfg.hidden,), "wqkv": ((cfg.Hq + 2 * cfg.Hkv) * cfg.d, cfg.hidden),
            "wo": (cfg.hidden, cfg.Hq * cfg.d), "ln2": (cfg.hidden,), "wgu": (2 * cfg.inter, cfg.hidden),
            "wd": (cfg.hidden, cfg.inter)}


def _weights(w: dict) -> LayerWeights:
    return LayerWeights(*[_ptr(w[n]) for n in LAYER_WEIGHTS])


def dualkv_layer_workspace_bytes(cfg: LayerConfig, groups) -> int:
    G, Ps, Ns, Rs = _groups(groups)
    return int(lib.dualkv_layer_workspace_bytes(ctypes.byref(cfg), G, Ps, Ns, Rs))


def dualkv_layer_fwd(cfg: LayerConfig, weights: dict, x, groups, y, workspace, stream=None, check: bool = True) -> int:
    """Calls dualkv_layer_fwd (x, y [T, hidden] bf16; weights: dict of bf16 device tensors)."""
    G, Ps, Ns, Rs = _groups(groups)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.dualkv_layer_fwd(ctypes.byref(cfg), ctypes.byref(_weights(weights)), _ptr(x), G, Ps, Ns, Rs, _ptr(y),
                              _ptr(workspace), nbytes, _stream(stream))
    if check:
        _check(st, "dualkv_layer_fwd")
    return st


def dualkv_layer_bwd(cfg: LayerConfig, weights: dict, x, dy, groups, dx, grads: dict, workspace, stream=None,
                     check: bool = True) -> int:
    """Calls dualkv_layer_bwd (grads: dict of fp32 device tensors, overwritten)."""
    G, Ps, Ns, Rs = _groups(groups)
    nbytes = workspace.numel() * workspace.element_size()
    g = LayerGrads(*[_ptr(grads[n]) for n in LAYER_WEIGHTS])
    st = lib.dualkv_layer_bwd(ctypes.byref(cfg), ctypes.byref(_weights(weights)), _ptr(x), _ptr(dy), G, Ps, Ns, Rs,
                              _ptr(dx), ctypes.byref(g), _ptr(workspace), nbytes, _stream(stream))
    if check:
        _check(st, "dualkv_layer_bwd")
    return st


def dualkv_packed_positions(groups):
    """Position id of every packed row (host list)."""
    G, Ps, Ns, Rs = _groups(groups)
    T = sum(int(p) + sum(int(r) for r in rs) for p, rs in groups)
    out = (ctypes.c_int32 * max(T, 1))()
    _check(lib.dualkv_packed_positions(G, Ps, Ns, Rs, out, T), "dualkv_packed_positions")
    return list(out[:T])


class PackedLayer:
    """Forward/backward of one packed decoder layer through the C ABI, with
    the workspace kept between the two calls."""

    def __init__(self, cfg: LayerConfig, weights: dict, groups):
        self.cfg, self.weights, self.groups = cfg, weights, [(int(p), tuple(int(r) for r in rs)) for p, rs in groups]
        dev = weights["wqkv"].device
        self.workspace = torch.empty(max(1, dualkv_layer_workspace_bytes(cfg, self.groups)), dtype=torch.uint8,
                                     device=dev)

    def forward(self, x, stream=None):
        y = torch.empty_like(x)
        dualkv_layer_fwd(self.cfg, self.weights, x, self.groups, y, self.workspace, stream)
        return y

    def backward(self, x, dy, stream=None):
        dx = torch.empty_like(x)
        grads = {n: torch.empty(t.shape, dtype=torch.float32, device=t.device) for n, t in self.weights.items()}
        dualkv_layer_bwd(self.cfg, self.weights, x, dy, self.groups, dx, grads, self.workspace, stream)
        return dx, grads


# --------------------------------------------------------------------------- autograd

class DualKVAttention(torch.autograd.Function):
    """torch.autograd wrapper of dualkv_fwd_groups / dualkv_bwd_groups.

    forward(q, k, v, groups, softmax_scale, deterministic, num_splits) -> out;
    the saved tensors are q, k, v, out and lse.  The backward's dout is made
    contiguous before the call (the library's layouts are dense)."""

    @staticmethod
    def forward(ctx, q, k, v, groups, softmax_scale, deterministic, num_splits):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, lse = forward_groups(q, k, v, groups, softmax_scale)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.groups, ctx.scale = groups, softmax_scale
        ctx.deterministic, ctx.num_splits = deterministic, num_splits
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = backward_groups(q, k, v, out, dout.contiguous(), lse, ctx.groups, ctx.scale,
                                     deterministic=ctx.deterministic, num_splits=ctx.num_splits)
        return dq, dk, dv, None, None, None, None


def dualkv_attention(q, k, v, P: Optional[int] = None, R_lens: Optional[Sequence[int]] = None, groups=None,
                     softmax_scale: Optional[float] = None, deterministic: bool = False, num_splits: int = 0):
    """Differentiable shared-prompt attention on packed rows.

    Give either (P, R_lens) for one prompt group or ``groups`` = [(P_g,
    R_lens_g), ...] for several.  q [T, Hq, d], k/v [T, Hkv, d] bf16 on the GPU;
    returns out [T, Hq, d].  The gradient reaching a prompt row of out is the
    gradient of the one shared row (its sequences' sum)."""
    if groups is None:
        if P is None or R_lens is None:
            raise ValueError("give (P, R_lens) or groups")
        groups = [(int(P), tuple(int(r) for r in R_lens))]
    else:
        groups = [(int(p), tuple(int(r) for r in rs)) for p, rs in groups]
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** -0.5
    return DualKVAttention.apply(q, k, v, groups, float(softmax_scale), bool(deterministic), int(num_splits))
