"""ctypes binding of libsn's C ABI (``include/sn_abi.h``).

Functions carry the C names and arguments.  They only marshal arguments:
tensors become raw device pointers, ``None`` becomes NULL, streams become
``cudaStream_t`` handles.  Every computation happens inside libsn's CUDA
kernels.  There is no fallback: if ``libsn.so`` is missing or fails to load,
importing the compute functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsn.so")

# --- constants mirrored from include/sn_abi.h
SN_ABI_VERSION_MAJOR, SN_ABI_VERSION_MINOR, SN_ABI_VERSION_PATCH = 1, 0, 0
SN_OK, SN_E_INVAL, SN_E_NOMEM, SN_E_IO, SN_E_FORMAT, SN_E_UNSUPPORTED, SN_E_DEVICE, SN_E_TIMEOUT = (
    0, -1, -2, -3, -4, -5, -6, -7)
SN_E_RANGE = -8
SN_CAP_SCAN_FMA, SN_CAP_SCAN_GATED, SN_CAP_RECUR_DIAG, SN_CAP_RECUR_DELTA = 1, 2, 4, 8
SN_CAP_RECUR_RWKV7, SN_CAP_DECODE, SN_CAP_SCAN_LOOKBACK, SN_CAP_SCAN_BACKWARD = 16, 32, 64, 128
SN_CAP_RECUR_CHUNKED, SN_CAP_READOUT, SN_CAP_DELTA_CHUNKED = 256, 512, 1024
SN_DECAY_PER_KEY, SN_DECAY_PER_HEAD, SN_DECAY_PER_KEY_GATED, SN_DECAY_PER_HEAD_GATED = 0, 1, 2, 3
SN_OPT_SCAN_KERNEL, SN_OPT_WAIT_LIMIT_US, SN_OPT_DEBUG_POISON, SN_OPT_LOOKBACK_CHUNK, SN_OPT_RECUR_KERNEL = (
    1, 2, 3, 4, 5)
SN_OPT_RECUR_TILE = 6
SN_OPT_DELTA_SEGMENTS = 7
SN_SCAN_KERNEL_AUTO, SN_SCAN_KERNEL_SEQUENTIAL, SN_SCAN_KERNEL_LOOKBACK, SN_SCAN_KERNEL_REDUCE_SCAN = 0, 1, 2, 3
SN_SCAN_KERNEL_FUSED = 4
SN_OP_SCAN_FMA, SN_OP_SCAN_GATED = 1, 2

# every symbol the header declares
EXPORTS = (
    "sn_abi_version", "sn_abi_check", "sn_abi_caps", "sn_status_str",
    "sn_ctx_create", "sn_ctx_free", "sn_ctx_set_workspace", "sn_workspace_bytes",
    "sn_ctx_last_error", "sn_ctx_set_option", "sn_ctx_get_option",
    "sn_scan_fma", "sn_scan_gated", "sn_scan_fma_backward", "sn_scan_gated_backward",
    "sn_recur_diag", "sn_recur_delta", "sn_recur_rwkv7", "sn_scan_lookback_noalloc",
    "sn_scan_host_staging_bytes", "sn_scan_host",
    "sn_recur_diag_chunked", "sn_recur_chunked_workspace_bytes", "sn_readout_norm_gate", "sn_readout_dskip",
    "sn_recur_delta_chunked", "sn_recur_delta_chunked_workspace_bytes",
)
SN_NOALLOC_MAX_TILES = 40960

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsn.so and declare the signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is not built; run scan_runtime_gb300.build() "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        i32, i64, u32, f32, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p
        sig = {
            "sn_abi_version": ([], u32),
            "sn_abi_check": ([i32], i32),
            "sn_abi_caps": ([], u32),
            "sn_status_str": ([i32], ctypes.c_char_p),
            "sn_ctx_create": ([i32, ctypes.POINTER(p)], i32),
            "sn_ctx_free": ([p], None),
            "sn_ctx_set_workspace": ([p, p, i64], i32),
            "sn_workspace_bytes": ([i32, i32, i32, i32], i64),
            "sn_ctx_last_error": ([p], i32),
            "sn_ctx_set_option": ([p, i32, i32], i32),
            "sn_ctx_get_option": ([p, i32, ctypes.POINTER(i32)], i32),
            "sn_scan_fma": ([p, i32, i32, i32, p, p, p, p, p, p], i32),
            "sn_scan_gated": ([p, i32, i32, i32, p, p, p, p, p, p], i32),
            "sn_scan_fma_backward": ([p, i32, i32, i32] + [p] * 9, i32),
            "sn_scan_gated_backward": ([p, i32, i32, i32] + [p] * 10, i32),
            "sn_recur_diag": ([p, i32, i32, i32, i32, i32, i32, i32, f32, p, p, p, p, p, p, p, p], i32),
            "sn_recur_delta": ([p, i32, i32, i32, i32, i32, f32, p, p, p, p, p, p, p, p], i32),
            "sn_recur_rwkv7": ([p, i32, i32, i32, i32, i32, p, p, p, p, p, p, p, p], i32),
            "sn_scan_lookback_noalloc": ([i32, i32, i32, i32, p, p, p, p, p, p, p], i32),
            "sn_scan_host_staging_bytes": ([i32, i32, i32, i32, i32], i64),
            "sn_scan_host": ([p, i32, i32, i32, i32] + [p] * 9 + [i64, p], i32),
            "sn_recur_diag_chunked": ([p, i32, i32, i32, i32, i32, i32, i32, f32, p, p, p, p, p, p, p, p], i32),
            "sn_recur_chunked_workspace_bytes": ([i32, i32, i32, i32, i32], i64),
            "sn_readout_norm_gate": ([p, i32, i32, i32, i32, p, p, p, f32, p, p], i32),
            "sn_readout_dskip": ([p, i32, i32, i32, i32, p, p, p, p, p], i32),
            "sn_recur_delta_chunked": ([p, i32, i32, i32, i32, i32, f32, p, p, p, p, p, p, p, p], i32),
            "sn_recur_delta_chunked_workspace_bytes": ([i32, i32, i32, i32, i32], i64),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def ptr(x) -> int | None:
    """Address of a tensor's data (device or host) or an int address; None stays NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensors passed to libsn must be contiguous")
    return x.data_ptr()


def stream_handle(stream) -> int | None:
    """cudaStream_t of a torch stream; None means torch's current stream."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


# ------------------------------------------------------------------ meta
def sn_abi_version() -> int:
    return load().sn_abi_version()


def sn_abi_check(major: int) -> int:
    return load().sn_abi_check(major)


def sn_abi_caps() -> int:
    return load().sn_abi_caps()


def sn_status_str(s: int) -> str:
    return load().sn_status_str(s).decode()


# ------------------------------------------------------------------ context
def sn_ctx_create(device: int):
    """Returns (status, handle)."""
    h = ctypes.c_void_p()
    s = load().sn_ctx_create(device, ctypes.byref(h))
    return s, h


def sn_ctx_free(ctx) -> None:
    load().sn_ctx_free(ctx)


def sn_ctx_set_workspace(ctx, ws, nbytes: int) -> int:
    return load().sn_ctx_set_workspace(ctx, ptr(ws), nbytes)


def sn_workspace_bytes(op: int, B: int, T: int, N: int) -> int:
    return load().sn_workspace_bytes(op, B, T, N)


def sn_ctx_last_error(ctx) -> int:
    return load().sn_ctx_last_error(ctx)


def sn_ctx_set_option(ctx, key: int, value: int) -> int:
    return load().sn_ctx_set_option(ctx, key, value)


def sn_ctx_get_option(ctx, key: int):
    """Returns (status, value)."""
    v = ctypes.c_int32()
    s = load().sn_ctx_get_option(ctx, key, ctypes.byref(v))
    return s, v.value


# ------------------------------------------------------------------ compute
def sn_scan_fma(ctx, B, T, N, a, b, s0, s_final, s_out, stream=None) -> int:
    return load().sn_scan_fma(ctx, B, T, N, ptr(a), ptr(b), ptr(s0), ptr(s_final), ptr(s_out),
                              stream_handle(stream))


def sn_scan_gated(ctx, B, T, N, a, u, s0, s_final, s_out, stream=None) -> int:
    return load().sn_scan_gated(ctx, B, T, N, ptr(a), ptr(u), ptr(s0), ptr(s_final), ptr(s_out),
                                stream_handle(stream))


def sn_scan_fma_backward(ctx, B, T, N, a, s0, s, grad_s, grad_final, grad_a, grad_b, grad_s0, stream=None) -> int:
    return load().sn_scan_fma_backward(ctx, B, T, N, ptr(a), ptr(s0), ptr(s), ptr(grad_s), ptr(grad_final),
                                       ptr(grad_a), ptr(grad_b), ptr(grad_s0), stream_handle(stream))


def sn_scan_gated_backward(ctx, B, T, N, a, u, s0, s, grad_s, grad_final, grad_a, grad_u, grad_s0,
                           stream=None) -> int:
    return load().sn_scan_gated_backward(ctx, B, T, N, ptr(a), ptr(u), ptr(s0), ptr(s), ptr(grad_s),
                                         ptr(grad_final), ptr(grad_a), ptr(grad_u), ptr(grad_s0),
                                         stream_handle(stream))


def sn_recur_diag(ctx, B, T, H, G, dk, dv, decay_kind, scale, q, k, v, d, S_in, S_out, o, stream=None) -> int:
    return load().sn_recur_diag(ctx, B, T, H, G, dk, dv, decay_kind, scale, ptr(q), ptr(k), ptr(v), ptr(d),
                                ptr(S_in), ptr(S_out), ptr(o), stream_handle(stream))


def sn_recur_delta(ctx, B, T, H, dk, dv, scale, q, k, v, beta, S_in, S_out, o, stream=None) -> int:
    return load().sn_recur_delta(ctx, B, T, H, dk, dv, scale, ptr(q), ptr(k), ptr(v), ptr(beta), ptr(S_in),
                                 ptr(S_out), ptr(o), stream_handle(stream))


def sn_recur_rwkv7(ctx, B, T, H, dk, dv, q, k, v, w, S_in, S_out, o, stream=None) -> int:
    return load().sn_recur_rwkv7(ctx, B, T, H, dk, dv, ptr(q), ptr(k), ptr(v), ptr(w), ptr(S_in), ptr(S_out),
                                 ptr(o), stream_handle(stream))


def sn_scan_lookback_noalloc(gated, B, T, N, a, b, s0, s_final, s_out, status_out=None, stream=None) -> int:
    return load().sn_scan_lookback_noalloc(gated, B, T, N, ptr(a), ptr(b), ptr(s0), ptr(s_final), ptr(s_out),
                                           ptr(status_out), stream_handle(stream))


def sn_scan_host_staging_bytes(B, T, N, forms_mask, rows_per_chunk) -> int:
    return load().sn_scan_host_staging_bytes(B, T, N, forms_mask, rows_per_chunk)


def sn_scan_host(ctx, B, T, N, rows_per_chunk, a, b, u, s0, s_out_fma, s_final_fma, s_out_gated, s_final_gated,
                 staging, staging_bytes, stream=None) -> int:
    return load().sn_scan_host(ctx, B, T, N, rows_per_chunk, ptr(a), ptr(b), ptr(u), ptr(s0), ptr(s_out_fma),
                               ptr(s_final_fma), ptr(s_out_gated), ptr(s_final_gated), ptr(staging), staging_bytes,
                               stream_handle(stream))


def sn_recur_diag_chunked(ctx, B, T, H, G, dk, dv, decay_kind, scale, q, k, v, d, S_in, S_out, o,
                          stream=None) -> int:
    return load().sn_recur_diag_chunked(ctx, B, T, H, G, dk, dv, decay_kind, scale, ptr(q), ptr(k), ptr(v),
                                        ptr(d), ptr(S_in), ptr(S_out), ptr(o), stream_handle(stream))


def sn_recur_chunked_workspace_bytes(B, T, H, dk, dv) -> int:
    return load().sn_recur_chunked_workspace_bytes(B, T, H, dk, dv)


def sn_readout_norm_gate(ctx, B, T, H, dv, o, g, w, eps, y, stream=None) -> int:
    return load().sn_readout_norm_gate(ctx, B, T, H, dv, ptr(o), ptr(g), ptr(w), eps, ptr(y), stream_handle(stream))


def sn_readout_dskip(ctx, B, T, H, dv, o, x, D, y, stream=None) -> int:
    return load().sn_readout_dskip(ctx, B, T, H, dv, ptr(o), ptr(x), ptr(D), ptr(y), stream_handle(stream))


def sn_recur_delta_chunked(ctx, B, T, H, dk, dv, scale, q, k, v, beta, S_in, S_out, o, stream=None) -> int:
    return load().sn_recur_delta_chunked(ctx, B, T, H, dk, dv, scale, ptr(q), ptr(k), ptr(v), ptr(beta), ptr(S_in),
                                         ptr(S_out), ptr(o), stream_handle(stream))


def sn_recur_delta_chunked_workspace_bytes(B, T, H, dk, dv) -> int:
    return load().sn_recur_delta_chunked_workspace_bytes(B, T, H, dk, dv)
