"""ctypes binding of libcf (include/cf.h): the same entry points under the same
names, plus thin conveniences that allocate outputs and workspaces with torch.

Argument marshalling only: every step of the computation runs in libcf's CUDA
kernels.  Loading fails loudly if libcf.so has not been built; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcf.so")

CF_OK = 0
CF_ERR_INVALID_ARG = 1
CF_ERR_UNSUPPORTED = 2
CF_ERR_MISALIGNED = 3
CF_ERR_WORKSPACE_TOO_SMALL = 4
CF_ERR_NOT_RESIDENT = 5
CF_ERR_CUDA = 6
CF_ERR_DEVICE_TIMEOUT = 7
CF_ERR_DEVICE_BOUNDS = 8
CF_ERR_NO_DEVICE = 9

CF_ACT_NONE = 0
CF_ACT_GELU_TANH = 1


class cf_tuning(ctypes.Structure):
    _fields_ = [
        ("n_slice", ctypes.c_int32),
        ("cluster_size", ctypes.c_int32),
        ("peer_max", ctypes.c_int32),
        ("max_clusters", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("stitch_mapping", ctypes.c_int32),
        ("timeout_us", ctypes.c_uint32),
        ("extra_arrivals", ctypes.c_int32),
        ("cluster_m", ctypes.c_int32),
        ("disable_pdl", ctypes.c_int32),
        ("trace", ctypes.c_void_p),
    ]


CF_TRACE_TILES = 16
CF_TRACE_EVENTS = 12
CF_TRACE_SLOTS = 4 + CF_TRACE_TILES * CF_TRACE_EVENTS
TRACE_EVENT_NAMES = ["tma_first", "tma_last", "mma_acc_free", "mma_first", "mma_done", "mma_wait_ns",
                     "epi_start", "epi_stats", "epi_cta", "epi_cluster", "epi_global", "epi_stored"]
# cf_trace_event (fused GEMM) and cf_trb_event (back-to-back GEMM) slots
(CF_TR_TMA_FIRST, CF_TR_TMA_LAST, CF_TR_MMA_ACC_FREE, CF_TR_MMA_FIRST, CF_TR_MMA_DONE, CF_TR_MMA_WAIT_NS,
 CF_TR_EPI_START, CF_TR_EPI_STATS, CF_TR_EPI_CTA, CF_TR_EPI_CLUSTER, CF_TR_EPI_GLOBAL, CF_TR_EPI_STORED) = range(12)
(CF_TRB_TMA_FIRST, CF_TRB_ML1_FIRST, CF_TRB_ML1_DONE, CF_TRB_EPI1_START, CF_TRB_EPI1_LOCAL, CF_TRB_EPI1_DONE,
 CF_TRB_ML2_START, CF_TRB_ML2_DONE, CF_TRB_EPI2_START, CF_TRB_EPI2_SENT, CF_TRB_EPI2_RECV,
 CF_TRB_EPI2_STORED) = range(12)


class cf_plan(ctypes.Structure):
    _fields_ = [
        ("n_slice", ctypes.c_int32),
        ("ctas_per_row", ctypes.c_int32),
        ("cluster_size", ctypes.c_int32),
        ("groups", ctypes.c_int32),
        ("leader_mode", ctypes.c_int32),
        ("row_blocks", ctypes.c_int32),
        ("clusters", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("cluster_m", ctypes.c_int32),
        ("staging_buffers", ctypes.c_int32),
    ]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class CfError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})"
                         + (f", cudaError {cf_last_cuda_error()}" if status == CF_ERR_CUDA else ""))


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_ST = ctypes.c_int

# name -> (restype, argtypes)
_SIGS = {
    "cf_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "cf_version": (ctypes.c_int, []),
    "cf_last_cuda_error": (ctypes.c_int, []),
    "cf_tuning_default": (None, [ctypes.POINTER(cf_tuning)]),
    "cf_plan_gemm_fused": (_ST, [_I64, _I64, _I64, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(cf_tuning), ctypes.POINTER(cf_plan)]),
    "cf_query_gemm_fused_plan": (_ST, [_I64, _I64, _I64, ctypes.c_int32, ctypes.POINTER(cf_tuning),
                                       ctypes.POINTER(cf_plan), ctypes.POINTER(ctypes.c_int32)]),
    "cf_gemm_fused_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "cf_stitch_workspace_size": (_SZ, [_I64, _I64]),
    "cf_workspace_init": (_ST, [_P, _SZ, _P]),
    "cf_get_device_status": (_ST, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "cf_gemm_fused_rownorm": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                    _P, _SZ, _P]),
    "cf_gemm_fused_rownorm_ex": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                       _P, _SZ, _P, ctypes.POINTER(cf_tuning)]),
    "cf_gemm_fused_rownorm_noalloc": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                            _P]),
    "cf_gemm_fused_rownorm_noalloc_status": (_ST, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "cf_gemm_fused_rmsnorm": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                    _P, _SZ, _P]),
    "cf_gemm_fused_rmsnorm_ex": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                       _P, _SZ, _P, ctypes.POINTER(cf_tuning)]),
    "cf_gemm_fused_residual_norm": (_ST, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                          ctypes.c_int, _P, _SZ, _P]),
    "cf_gemm_fused_residual_norm_ex": (_ST, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                             ctypes.c_int, _P, _SZ, _P, ctypes.POINTER(cf_tuning)]),
    "cf_gemm_fused_rowsoftmax_causal": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _F, _I64, _P, _SZ, _P]),
    "cf_gemm_fused_rowsoftmax_causal_ex": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _F, _I64, _P, _SZ, _P,
                                                 ctypes.POINTER(cf_tuning)]),
    "cf_gemm_fused_rowsoftmax": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _F, _P, _SZ, _P]),
    "cf_gemm_fused_rowsoftmax_ex": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _F, _P, _SZ, _P,
                                          ctypes.POINTER(cf_tuning)]),
    "cf_unfused_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "cf_unfused_gemm_rownorm": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                      _P, _SZ, _P]),
    "cf_unfused_gemm_rmsnorm": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                      _P, _SZ, _P]),
    "cf_unfused_gemm_residual_norm": (_ST, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                            ctypes.c_int, _P, _SZ, _P]),
    "cf_unfused_gemm_rowsoftmax": (_ST, [_P, _P, _P, _P, _I64, _I64, _I64, _F, _P, _SZ, _P]),
    "cf_b2b_workspace_size": (_SZ, []),
    "cf_query_b2b_plan": (_ST, [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(cf_tuning),
                                ctypes.POINTER(cf_plan)]),
    "cf_b2b_gemm": (_ST, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F, ctypes.c_int, _P, _SZ, _P]),
    "cf_b2b_gemm_ex": (_ST, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F, ctypes.c_int, _P, _SZ, _P,
                             ctypes.POINTER(cf_tuning)]),
    "cf_b2b_gemm_layernorm": (_ST, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F, _F, _P, _SZ, _P]),
    "cf_b2b_gemm_layernorm_ex": (_ST, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _F, _F, _P, _SZ, _P,
                                       ctypes.POINTER(cf_tuning)]),
    "cf_stitch_add_layernorm": (_ST, [_P, _P, _P, _P, _P, _I64, _I64, _F, _P, _SZ, _P]),
    "cf_stitch_add_layernorm_ex": (_ST, [_P, _P, _P, _P, _P, _I64, _I64, _F, _P, _SZ, _P,
                                         ctypes.POINTER(cf_tuning)]),
    "cf_stitch_batchnorm_workspace_size": (_SZ, [_I64, _I64]),
    "cf_stitch_batchnorm": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, _SZ, _P]),
    "cf_stitch_batchnorm_ex": (_ST, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, _SZ, _P,
                                     ctypes.POINTER(cf_tuning)]),
    "cf_query_stitch_batchnorm_plan": (_ST, [_I64, _I64, ctypes.POINTER(cf_tuning), ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32)]),
    "cf_stitch_rowreduce_broadcast": (_ST, [_P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "cf_stitch_rowreduce_broadcast_ex": (_ST, [_P, _P, _P, _I64, _I64, _P, _SZ, _P,
                                               ctypes.POINTER(cf_tuning)]),
    "cf_stitch_powadd_softmax": (_ST, [_P, _P, _F, _P, _I64, _I64, _P, _SZ, _P]),
    "cf_stitch_powadd_softmax_ex": (_ST, [_P, _P, _F, _P, _I64, _I64, _P, _SZ, _P, ctypes.POINTER(cf_tuning)]),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libcf.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libcf.so not built at {LIB_PATH}; run "
                                  "`python -m memory_fusion_gb300.build` (no fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def declared_symbols():
    return list(_SIGS)


# ---------------------------------------------------------------------------
# raw entry points (same names and argument order as the C ABI)
# ---------------------------------------------------------------------------
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _tun(t):
    return None if t is None else ctypes.byref(t)


def status_string(status: int) -> str:
    return lib().cf_status_string(int(status)).decode()


def cf_version() -> int:
    return lib().cf_version()


def cf_last_cuda_error() -> int:
    return lib().cf_last_cuda_error()


def cf_tuning_default() -> cf_tuning:
    t = cf_tuning()
    lib().cf_tuning_default(ctypes.byref(t))
    return t


def cf_plan_gemm_fused(M, N, K, sm_count, max_active_clusters, tuning=None):
    """max_active_clusters: 17 ints, index = cluster size (entry 0 unused)."""
    if len(max_active_clusters) != 17:
        raise ValueError("max_active_clusters needs 17 entries (index = cluster size)")
    arr = (ctypes.c_int32 * 17)(*[int(v) for v in max_active_clusters])
    p = cf_plan()
    st = lib().cf_plan_gemm_fused(M, N, K, sm_count, arr, _tun(tuning), ctypes.byref(p))
    return st, p


def cf_query_gemm_fused_plan(M, N, K, kind, tuning=None):
    """(status, plan, max_active_clusters[17]) on the current device; kind 0 LN, 1 GELU+LN, 2 softmax."""
    p = cf_plan()
    arr = (ctypes.c_int32 * 17)()
    st = lib().cf_query_gemm_fused_plan(M, N, K, kind, _tun(tuning), ctypes.byref(p), arr)
    return st, p, list(arr)


def cf_gemm_fused_workspace_size(M, N, K) -> int:
    return lib().cf_gemm_fused_workspace_size(M, N, K)


def cf_stitch_workspace_size(rows, cols) -> int:
    return lib().cf_stitch_workspace_size(rows, cols)


def cf_workspace_init(ws, nbytes, stream=None) -> int:
    return lib().cf_workspace_init(_ptr(ws), nbytes, _stream(stream))


def cf_get_device_status(ws, stream=None):
    info = ctypes.c_int32(0)
    st = lib().cf_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(info))
    return st, info.value


def cf_gemm_fused_rownorm(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, workspace,
                          workspace_bytes, stream=None, tuning=None) -> int:
    L = lib()
    if tuning is None:
        return L.cf_gemm_fused_rownorm(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                       M, N, K, alpha, eps, act, _ptr(workspace), workspace_bytes,
                                       _stream(stream))
    return L.cf_gemm_fused_rownorm_ex(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                      M, N, K, alpha, eps, act, _ptr(workspace), workspace_bytes,
                                      _stream(stream), _tun(tuning))


def cf_gemm_fused_rmsnorm(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, workspace,
                          workspace_bytes, stream=None, tuning=None) -> int:
    """Y = RMSNorm(act(alpha*X.W + bias)) * gamma (+ beta); beta may be None."""
    L = lib()
    if tuning is None:
        return L.cf_gemm_fused_rmsnorm(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                       M, N, K, alpha, eps, act, _ptr(workspace), workspace_bytes,
                                       _stream(stream))
    return L.cf_gemm_fused_rmsnorm_ex(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                      M, N, K, alpha, eps, act, _ptr(workspace), workspace_bytes,
                                      _stream(stream), _tun(tuning))


CF_NORM_LAYER = 0
CF_NORM_RMS = 1


def cf_gemm_fused_residual_norm(X, W, bias, R, gamma, beta, Y, M, N, K, alpha, eps, act, norm, workspace,
                                workspace_bytes, stream=None, tuning=None) -> int:
    """Y = Norm(act(alpha*X.W + bias) + R) * gamma (+ beta); norm CF_NORM_LAYER or CF_NORM_RMS."""
    L = lib()
    if tuning is None:
        return L.cf_gemm_fused_residual_norm(_ptr(X), _ptr(W), _ptr(bias), _ptr(R), _ptr(gamma), _ptr(beta),
                                             _ptr(Y), M, N, K, alpha, eps, act, norm, _ptr(workspace),
                                             workspace_bytes, _stream(stream))
    return L.cf_gemm_fused_residual_norm_ex(_ptr(X), _ptr(W), _ptr(bias), _ptr(R), _ptr(gamma), _ptr(beta),
                                            _ptr(Y), M, N, K, alpha, eps, act, norm, _ptr(workspace),
                                            workspace_bytes, _stream(stream), _tun(tuning))


def cf_unfused_gemm_residual_norm(X, W, bias, R, gamma, beta, Y, M, N, K, alpha, eps, act, norm, workspace,
                                  workspace_bytes, stream=None) -> int:
    return lib().cf_unfused_gemm_residual_norm(_ptr(X), _ptr(W), _ptr(bias), _ptr(R), _ptr(gamma), _ptr(beta),
                                               _ptr(Y), M, N, K, alpha, eps, act, norm, _ptr(workspace),
                                               workspace_bytes, _stream(stream))


def cf_gemm_fused_rownorm_noalloc(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, stream=None) -> int:
    """cf_gemm_fused_rownorm without a workspace: for callers that cannot
    allocate device memory; its scratch is a fixed 4 MiB array inside libcf."""
    return lib().cf_gemm_fused_rownorm_noalloc(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                               M, N, K, alpha, eps, act, _stream(stream))


def cf_gemm_fused_rownorm_noalloc_status(stream=None):
    """(status, info) of the no-allocation calls on the current device: waits
    for the stream, reads and clears the fixed scratch array's error word."""
    info = ctypes.c_int32(0)
    st = lib().cf_gemm_fused_rownorm_noalloc_status(_stream(stream), ctypes.byref(info))
    return st, info.value


def cf_gemm_fused_rowsoftmax(X, W, bias, Y, M, N, K, scale, workspace, workspace_bytes,
                             stream=None, tuning=None) -> int:
    L = lib()
    if tuning is None:
        return L.cf_gemm_fused_rowsoftmax(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), M, N, K, scale,
                                          _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_gemm_fused_rowsoftmax_ex(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), M, N, K, scale,
                                         _ptr(workspace), workspace_bytes, _stream(stream), _tun(tuning))


def cf_stitch_rowreduce_broadcast(A, row_bias, out, rows, cols, workspace, workspace_bytes,
                                  stream=None, tuning=None) -> int:
    L = lib()
    if tuning is None:
        return L.cf_stitch_rowreduce_broadcast(_ptr(A), _ptr(row_bias), _ptr(out), rows, cols,
                                               _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_stitch_rowreduce_broadcast_ex(_ptr(A), _ptr(row_bias), _ptr(out), rows, cols,
                                              _ptr(workspace), workspace_bytes, _stream(stream),
                                              _tun(tuning))


def cf_stitch_powadd_softmax(A, w, p, out, rows, cols, workspace, workspace_bytes, stream=None, tuning=None) -> int:
    L = lib()
    if tuning is None:
        return L.cf_stitch_powadd_softmax(_ptr(A), _ptr(w), p, _ptr(out), rows, cols, _ptr(workspace),
                                          workspace_bytes, _stream(stream))
    return L.cf_stitch_powadd_softmax_ex(_ptr(A), _ptr(w), p, _ptr(out), rows, cols, _ptr(workspace),
                                         workspace_bytes, _stream(stream), _tun(tuning))


def cf_unfused_workspace_size(M, N, K) -> int:
    return lib().cf_unfused_workspace_size(M, N, K)


def cf_unfused_gemm_rownorm(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, workspace, workspace_bytes,
                            stream=None) -> int:
    """The unfused two-kernel composition (GEMM -> fp32 P -> row kernel), for comparison."""
    return lib().cf_unfused_gemm_rownorm(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                         M, N, K, alpha, eps, act, _ptr(workspace), workspace_bytes,
                                         _stream(stream))


def cf_gemm_fused_rowsoftmax_causal(X, W, bias, Y, M, N, K, scale, offset, workspace, workspace_bytes,
                                    stream=None, tuning=None) -> int:
    """Y = softmax over each row of scale*X.W + bias keeping column j of row i iff j <= i + offset."""
    L = lib()
    if tuning is None:
        return L.cf_gemm_fused_rowsoftmax_causal(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), M, N, K, scale, offset,
                                                 _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_gemm_fused_rowsoftmax_causal_ex(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), M, N, K, scale, offset,
                                                _ptr(workspace), workspace_bytes, _stream(stream), _tun(tuning))


def cf_unfused_gemm_rmsnorm(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, act, workspace, workspace_bytes,
                            stream=None) -> int:
    return lib().cf_unfused_gemm_rmsnorm(_ptr(X), _ptr(W), _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(Y),
                                         M, N, K, alpha, eps, act, _ptr(workspace), workspace_bytes,
                                         _stream(stream))


def cf_unfused_gemm_rowsoftmax(X, W, bias, Y, M, N, K, scale, workspace, workspace_bytes, stream=None) -> int:
    return lib().cf_unfused_gemm_rowsoftmax(_ptr(X), _ptr(W), _ptr(bias), _ptr(Y), M, N, K, scale,
                                            _ptr(workspace), workspace_bytes, _stream(stream))


CF_B2B_SOFTMAX = 0
CF_B2B_GELU_TANH = 1
CF_B2B_LAYERNORM = 2


def cf_b2b_workspace_size() -> int:
    return lib().cf_b2b_workspace_size()


def cf_query_b2b_plan(M, K, N1, N2, op, tuning=None):
    """(status, plan) of the back-to-back GEMM launch on the current device."""
    p = cf_plan()
    st = lib().cf_query_b2b_plan(M, K, N1, N2, op, _tun(tuning), ctypes.byref(p))
    return st, p


def cf_b2b_gemm(X, W1, b1, W2, O, M, K, N1, N2, alpha, op, workspace, workspace_bytes, stream=None,
                tuning=None) -> int:
    """O = bf16(F(alpha*X.W1 + b1)) . W2 with F the row softmax (op 0) or GELU_tanh (op 1)."""
    L = lib()
    if tuning is None:
        return L.cf_b2b_gemm(_ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(O), M, K, N1, N2, alpha, op,
                             _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_b2b_gemm_ex(_ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(O), M, K, N1, N2, alpha, op,
                            _ptr(workspace), workspace_bytes, _stream(stream), _tun(tuning))


def check(status: int, what: str = "libcf"):
    if status != CF_OK:
        raise CfError(status, what)


# ---------------------------------------------------------------------------
# conveniences over torch tensors (allocation in Python, compute in libcf)
# ---------------------------------------------------------------------------
def tuning(**kw) -> cf_tuning:
    t = cf_tuning_default()
    for k, v in kw.items():
        setattr(t, k, v.data_ptr() if k == "trace" and hasattr(v, "data_ptr") else v)
    return t


def new_workspace(nbytes: int, device=None, stream=None):
    import torch
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")
    check(cf_workspace_init(ws, ws.numel(), stream), "cf_workspace_init")
    return ws


def gemm_fused_rownorm(X, W, bias, gamma, beta, *, alpha=1.0, eps=1e-5, act="none", out=None,
                       workspace=None, stream=None, tuning=None):
    """Y = LayerNorm(act(alpha*X@W + bias))*gamma + beta; X, W bf16 CUDA tensors."""
    import torch
    M, K = X.shape
    N = W.shape[1]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = workspace if workspace is not None else new_workspace(cf_gemm_fused_workspace_size(M, N, K),
                                                               X.device, stream)
    a = {"none": CF_ACT_NONE, "gelu_tanh": CF_ACT_GELU_TANH}[act]
    check(cf_gemm_fused_rownorm(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, a, ws, ws.numel(),
                                stream, tuning), "cf_gemm_fused_rownorm")
    return Y


def gemm_fused_rmsnorm(X, W, bias, gamma, beta=None, *, alpha=1.0, eps=1e-5, act="none", out=None,
                       workspace=None, stream=None, tuning=None):
    """Y = RMSNorm(act(alpha*X@W + bias))*gamma (+ beta); X, W bf16 CUDA tensors."""
    import torch
    M, K = X.shape
    N = W.shape[1]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = workspace if workspace is not None else new_workspace(cf_gemm_fused_workspace_size(M, N, K),
                                                               X.device, stream)
    a = {"none": CF_ACT_NONE, "gelu_tanh": CF_ACT_GELU_TANH}[act]
    check(cf_gemm_fused_rmsnorm(X, W, bias, gamma, beta, Y, M, N, K, alpha, eps, a, ws, ws.numel(),
                                stream, tuning), "cf_gemm_fused_rmsnorm")
    return Y


def gemm_fused_rowsoftmax(X, W, bias=None, *, scale=1.0, out=None, workspace=None, stream=None,
                          tuning=None):
    """Y = softmax(scale*X@W + bias) over rows; X, W bf16 CUDA tensors."""
    import torch
    M, K = X.shape
    N = W.shape[1]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = workspace if workspace is not None else new_workspace(cf_gemm_fused_workspace_size(M, N, K),
                                                               X.device, stream)
    check(cf_gemm_fused_rowsoftmax(X, W, bias, Y, M, N, K, scale, ws, ws.numel(), stream, tuning),
          "cf_gemm_fused_rowsoftmax")
    return Y


def gemm_fused_residual_norm(X, W, bias, R, gamma, beta=None, *, alpha=1.0, eps=1e-5, act="none", norm="layer",
                             out=None, workspace=None, stream=None, tuning=None):
    """Y = Norm(act(alpha*X@W + bias) + R)*gamma (+ beta), Norm = "layer" or "rms"; X, W, R bf16 CUDA tensors."""
    import torch
    M, K = X.shape
    N = W.shape[1]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = workspace if workspace is not None else new_workspace(cf_gemm_fused_workspace_size(M, N, K),
                                                               X.device, stream)
    a = {"none": CF_ACT_NONE, "gelu_tanh": CF_ACT_GELU_TANH}[act]
    n = {"layer": CF_NORM_LAYER, "rms": CF_NORM_RMS}[norm]
    check(cf_gemm_fused_residual_norm(X, W, bias, R, gamma, beta, Y, M, N, K, alpha, eps, a, n, ws, ws.numel(),
                                      stream, tuning), "cf_gemm_fused_residual_norm")
    return Y


def gemm_fused_rowsoftmax_causal(X, W, bias=None, *, scale=1.0, offset=0, out=None, workspace=None, stream=None,
                                 tuning=None):
    """Y = softmax over each row of scale*X@W + bias keeping column j of row i iff j <= i + offset."""
    import torch
    M, K = X.shape
    N = W.shape[1]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = workspace if workspace is not None else new_workspace(cf_gemm_fused_workspace_size(M, N, K),
                                                               X.device, stream)
    check(cf_gemm_fused_rowsoftmax_causal(X, W, bias, Y, M, N, K, scale, offset, ws, ws.numel(), stream, tuning),
          "cf_gemm_fused_rowsoftmax_causal")
    return Y


def cf_b2b_gemm_layernorm(X, W1, b1, gamma1, beta1, W2, O, M, K, N1, N2, alpha, eps, workspace, workspace_bytes,
                          stream=None, tuning=None) -> int:
    """O = bf16(LayerNorm(alpha*X.W1 + b1)*gamma1 + beta1) . W2 (LayerNorm over the N1 columns)."""
    L = lib()
    if tuning is None:
        return L.cf_b2b_gemm_layernorm(_ptr(X), _ptr(W1), _ptr(b1), _ptr(gamma1), _ptr(beta1), _ptr(W2), _ptr(O),
                                       M, K, N1, N2, alpha, eps, _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_b2b_gemm_layernorm_ex(_ptr(X), _ptr(W1), _ptr(b1), _ptr(gamma1), _ptr(beta1), _ptr(W2), _ptr(O),
                                      M, K, N1, N2, alpha, eps, _ptr(workspace), workspace_bytes, _stream(stream),
                                      _tun(tuning))


def cf_stitch_add_layernorm(A, R, gamma, beta, out, rows, cols, eps, workspace, workspace_bytes, stream=None,
                            tuning=None) -> int:
    """out = LayerNorm(A + R) * gamma + beta over each row (R may be None)."""
    L = lib()
    if tuning is None:
        return L.cf_stitch_add_layernorm(_ptr(A), _ptr(R), _ptr(gamma), _ptr(beta), _ptr(out), rows, cols, eps,
                                         _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_stitch_add_layernorm_ex(_ptr(A), _ptr(R), _ptr(gamma), _ptr(beta), _ptr(out), rows, cols, eps,
                                        _ptr(workspace), workspace_bytes, _stream(stream), _tun(tuning))


def cf_stitch_batchnorm_workspace_size(rows, cols) -> int:
    return lib().cf_stitch_batchnorm_workspace_size(rows, cols)


def cf_stitch_batchnorm(A, gamma, beta, out, mean_out, var_out, rows, cols, eps, workspace, workspace_bytes,
                        stream=None, tuning=None) -> int:
    """out = (A - mean_col)/sqrt(var_col + eps)*gamma + beta with batch statistics over the rows."""
    L = lib()
    if tuning is None:
        return L.cf_stitch_batchnorm(_ptr(A), _ptr(gamma), _ptr(beta), _ptr(out), _ptr(mean_out), _ptr(var_out),
                                     rows, cols, eps, _ptr(workspace), workspace_bytes, _stream(stream))
    return L.cf_stitch_batchnorm_ex(_ptr(A), _ptr(gamma), _ptr(beta), _ptr(out), _ptr(mean_out), _ptr(var_out),
                                    rows, cols, eps, _ptr(workspace), workspace_bytes, _stream(stream), _tun(tuning))


def cf_query_stitch_batchnorm_plan(rows, cols, tuning=None):
    """(status, mapping 3 Regional / 4 Global, grid) on the current device."""
    m, g = ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().cf_query_stitch_batchnorm_plan(rows, cols, _tun(tuning), ctypes.byref(m), ctypes.byref(g))
    return st, m.value, g.value


def stitch_add_layernorm(A, R, gamma, beta, *, eps=1e-5, out=None, workspace=None, stream=None, tuning=None):
    """LayerNorm(A + R) * gamma + beta over rows; fp32 CUDA tensors (R may be None)."""
    import torch
    rows, cols = A.shape
    O = out if out is not None else torch.empty_like(A)
    ws = workspace if workspace is not None else new_workspace(cf_stitch_workspace_size(rows, cols), A.device,
                                                               stream)
    check(cf_stitch_add_layernorm(A, R, gamma, beta, O, rows, cols, eps, ws, ws.numel(), stream, tuning),
          "cf_stitch_add_layernorm")
    return O


def stitch_batchnorm(A, gamma, beta, *, eps=1e-5, out=None, workspace=None, stream=None, tuning=None):
    """(out, mean, var): BatchNorm of fp32 A [rows, cols] with its batch statistics."""
    import torch
    rows, cols = A.shape
    O = out if out is not None else torch.empty_like(A)
    mean = torch.empty(cols, dtype=torch.float32, device=A.device)
    var = torch.empty(cols, dtype=torch.float32, device=A.device)
    ws = workspace if workspace is not None else new_workspace(cf_stitch_batchnorm_workspace_size(rows, cols),
                                                               A.device, stream)
    check(cf_stitch_batchnorm(A, gamma, beta, O, mean, var, rows, cols, eps, ws, ws.numel(), stream, tuning),
          "cf_stitch_batchnorm")
    return O, mean, var


def b2b_gemm(X, W1, W2, b1=None, *, op="softmax", alpha=1.0, gamma1=None, beta1=None, eps=1e-5, out=None,
             workspace=None, stream=None, tuning=None):
    """O = bf16(F(alpha*X@W1 + b1)) @ W2, F = "softmax" (rows), "gelu_tanh" or "layernorm" (rows, with
    gamma1, beta1); bf16 CUDA tensors."""
    import torch
    ops = {"softmax": CF_B2B_SOFTMAX, "gelu_tanh": CF_B2B_GELU_TANH, "layernorm": CF_B2B_LAYERNORM}
    if op not in ops:
        raise ValueError(f"unknown op {op!r}")
    M, K = X.shape
    N1 = W1.shape[1]
    N2 = W2.shape[1]
    O = out if out is not None else torch.empty((M, N2), dtype=torch.bfloat16, device=X.device)
    ws = workspace if workspace is not None else new_workspace(cf_b2b_workspace_size(), X.device, stream)
    if op == "layernorm":
        check(cf_b2b_gemm_layernorm(X, W1, b1, gamma1, beta1, W2, O, M, K, N1, N2, alpha, eps, ws, ws.numel(),
                                    stream, tuning), "cf_b2b_gemm_layernorm")
    else:
        check(cf_b2b_gemm(X, W1, b1, W2, O, M, K, N1, N2, alpha, ops[op], ws, ws.numel(), stream, tuning),
              "cf_b2b_gemm")
    return O


def stitch_rowreduce_broadcast(A, row_bias, *, out=None, workspace=None, stream=None, tuning=None):
    """out = softmax_row(A^3 + row_bias[:, None]); fp32 CUDA tensors."""
    import torch
    rows, cols = A.shape
    O = out if out is not None else torch.empty_like(A)
    ws = workspace if workspace is not None else new_workspace(cf_stitch_workspace_size(rows, cols),
                                                               A.device, stream)
    check(cf_stitch_rowreduce_broadcast(A, row_bias, O, rows, cols, ws, ws.numel(), stream, tuning),
          "cf_stitch_rowreduce_broadcast")
    return O


def stitch_powadd_softmax(A, w, p, *, out=None, workspace=None, stream=None, tuning=None):
    """out = softmax_row(A + w[None, :] ** p) (w > 0); fp32 CUDA tensors."""
    import torch
    rows, cols = A.shape
    O = out if out is not None else torch.empty_like(A)
    ws = workspace if workspace is not None else new_workspace(cf_stitch_workspace_size(rows, cols),
                                                               A.device, stream)
    check(cf_stitch_powadd_softmax(A, w, float(p), O, rows, cols, ws, ws.numel(), stream, tuning),
          "cf_stitch_powadd_softmax")
    return O
