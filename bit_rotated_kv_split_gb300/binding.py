"""ctypes binding of liboscar.so (include/oscar.h): argument marshalling only.

Every function keeps the C name and forwards torch tensors as raw device or
host pointers; all computation happens inside the library.  Importing this
module loads the library and raises if it is missing - there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_double, c_float, c_int32, c_int64, c_size_t, c_void_p

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# the in-tree library; OSCAR_LIBRARY names another build of it (a
# verification build, for instance)
LIB_PATH = os.environ.get("OSCAR_LIBRARY") or os.path.join(_PKG, "liboscar.so")

OSCAR_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "ALIGNMENT", 3: "WORKSPACE", 4: "CUDA",
                5: "NO_CONVERGENCE", 6: "UNSUPPORTED", 7: "FILE"}
DEV_PAGE_BOUNDS, DEV_LENGTH, DEV_TIMEOUT = 0x1, 0x2, 0x4
OSCAR_STEP_OVERLAP_PREVIOUS = 0x1     # oscar_decode_step flag


class OscarError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, STATUS_NAMES.get(status, "?"), status))


class LayerDesc(ctypes.Structure):
    """Mirror of `oscar_layer_desc`."""
    _fields_ = [
        ("batch", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32), ("head_dim", c_int32),
        ("sink_cap", c_int32), ("recent_cap", c_int32), ("max_pages_per_seq", c_int32),
        ("max_hist", c_int32), ("n_pages", c_int64), ("tau_k", c_float), ("tau_v", c_float),
        ("pages", c_void_p), ("page_table", c_void_p), ("hist_len", c_void_p),
        ("sink_k", c_void_p), ("sink_v", c_void_p), ("sink_len", c_void_p),
        ("recent_k", c_void_p), ("recent_v", c_void_p), ("recent_len", c_void_p),
        ("recent_start", c_void_p), ("r_k", c_void_p), ("r_v", c_void_p), ("dev_status", c_void_p),
        ("quant_group_k", c_int32), ("quant_group_v", c_int32),
        ("codebook", c_int32), ("levels_k", c_float * 4), ("levels_v", c_float * 4),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("liboscar.so is not built (%s); run bit_rotated_kv_split_gb300.build" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sig = {
        "oscar_status_string": (ctypes.c_char_p, [c_int32]),
        "oscar_abi_version": (c_int32, []),
        "oscar_set_page_wait_limit": (c_int64, [c_int64]),
        "oscar_block_bytes": (c_int64, [c_int32, c_int32]),
        "oscar_build_rotation": (c_int32, [P, c_int64, c_int32, P, P]),
        "oscar_build_canalized_rotation": (c_int32, [c_int32, c_int32, P]),
        "oscar_build_rotation_from_covariance": (c_int32, [P, c_int32, P, P]),
        "oscar_covariance": (c_int32, [P, c_int64, c_int32, c_int64, P, P, ctypes.POINTER(c_size_t), P]),
        "oscar_value_covariance": (c_int32, [P, c_int64, P, P, c_int64, c_int32, c_int64, P, P,
                                             ctypes.POINTER(c_size_t), P]),
        "oscar_score_weighted_rows": (c_int32, [P, c_int64, P, P, c_int64, c_int32, c_double, P]),
        "oscar_clip_threshold": (c_int32, [P, c_int64, c_int32, c_int32, P, c_double, P]),
        "oscar_fit_codebook": (c_int32, [P, c_int64, c_int32, P, c_double, c_int32, P]),
        "oscar_rotation_file_write": (c_int32, [ctypes.c_char_p, c_int32, c_int32, c_int32, P, P, P, P]),
        "oscar_rotation_file_info": (c_int32, [ctypes.c_char_p, P, P, P]),
        "oscar_rotation_file_read": (c_int32, [ctypes.c_char_p, c_int32, c_int32, c_int32, P, P, P, P]),
        "oscar_quantize_append": (c_int32, [ctypes.POINTER(LayerDesc), P, P, c_int64, c_int64, P,
                                            P, P, c_int32, P, P, P]),
        "oscar_quantize_append_overlapped": (c_int32, [ctypes.POINTER(LayerDesc), P, P, c_int64, c_int64, P,
                                                       P, P, c_int32, P, P, P]),
        "oscar_decode_attention": (c_int32, [ctypes.POINTER(LayerDesc), P, P, P,
                                             ctypes.POINTER(c_size_t), P]),
        "oscar_decode_attention_static": (c_int32, [ctypes.POINTER(LayerDesc), P, P, P]),
        "oscar_decode_step": (c_int32, [ctypes.POINTER(LayerDesc), P, P, c_size_t, P, P, c_int64, c_int64, P, P,
                                        P, c_int32, P, P, P, P, P, c_size_t, P, ctypes.c_uint32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _check(fn, status):
    if status != OSCAR_OK:
        raise OscarError(fn, status)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def oscar_status_string(status: int) -> str:
    return lib.oscar_status_string(status).decode()


def oscar_abi_version() -> int:
    return lib.oscar_abi_version()


def oscar_set_page_wait_limit(limit_ns: int) -> int:
    """Limit of the decode kernel's waits for page copies (<= 0: the default, 1 s); returns the previous one."""
    return int(lib.oscar_set_page_wait_limit(int(limit_ns)))


def oscar_block_bytes(quant_group_k: int = 128, quant_group_v: int = 128) -> int:
    """Bytes of one (page, KV head) block of the pool; 0 for an invalid group size."""
    return lib.oscar_block_bytes(int(quant_group_k), int(quant_group_v))


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def oscar_build_rotation(x: np.ndarray):
    """(R [d][d], eigenvalues [d]) from calibration rows x [n][d] (host float64)."""
    x = _f64(x)
    n, d = x.shape
    r = np.empty((d, d), dtype=np.float64)
    w = np.empty(d, dtype=np.float64)
    _check("oscar_build_rotation", lib.oscar_build_rotation(x.ctypes.data, n, d, r.ctypes.data, w.ctypes.data))
    return r, w


def oscar_build_canalized_rotation(d: int, block: int):
    """Block-diagonal OScaR rotation R [d][d] (host float64)."""
    r = np.empty((d, d), dtype=np.float64)
    _check("oscar_build_canalized_rotation", lib.oscar_build_canalized_rotation(d, block, r.ctypes.data))
    return r


def oscar_build_rotation_from_covariance(c: np.ndarray):
    """(R [d][d], eigenvalues [d]) from a covariance c [d][d] (host float64)."""
    c = _f64(c)
    d = c.shape[0]
    r = np.empty((d, d), dtype=np.float64)
    w = np.empty(d, dtype=np.float64)
    _check("oscar_build_rotation_from_covariance",
           lib.oscar_build_rotation_from_covariance(c.ctypes.data, d, r.ctypes.data, w.ctypes.data))
    return r, w


def oscar_covariance_workspace_bytes(n: int) -> int:
    size = c_size_t(0)
    _check("oscar_covariance", lib.oscar_covariance(None, int(n), 128, 128, None, None, ctypes.byref(size), None))
    return size.value


def oscar_covariance(x, c_out, workspace, stream=None) -> None:
    """c_out [128][128] fp32 (device) = x^T x / n over the bf16 rows x [n][ld] (device)."""
    n, ld = int(x.shape[0]), int(x.stride(0))
    size = c_size_t(workspace.numel() * workspace.element_size())
    _check("oscar_covariance", lib.oscar_covariance(_ptr(x), n, 128, ld, _ptr(c_out), _ptr(workspace),
                                                    ctypes.byref(size), _stream(stream)))


def oscar_value_covariance_workspace_bytes(n_q: int) -> int:
    size = c_size_t(0)
    _check("oscar_value_covariance", lib.oscar_value_covariance(None, int(n_q), None, None, 1, 128, 128, None, None,
                                                                ctypes.byref(size), None))
    return size.value


def oscar_value_covariance(q, k, v, c_out, workspace, stream=None) -> None:
    """c_out [128][128] fp32 (device) = (S V)^T (S V) / n_q, S = softmax(q k^T / sqrt(128)),
    over bf16 rows q [n_q][ld], k, v [n_k][ld] (device, one row stride)."""
    n_q, n_k, ld = int(q.shape[0]), int(k.shape[0]), int(q.stride(0))
    if int(k.stride(0)) != ld or int(v.stride(0)) != ld or int(v.shape[0]) != n_k:
        raise ValueError("q, k and v must share one row stride; k and v one row count")
    size = c_size_t(workspace.numel() * workspace.element_size())
    _check("oscar_value_covariance", lib.oscar_value_covariance(
        _ptr(q), n_q, _ptr(k), _ptr(v), n_k, 128, ld, _ptr(c_out), _ptr(workspace), ctypes.byref(size),
        _stream(stream)))


def oscar_score_weighted_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float = None):
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[1]
    out = np.empty((q.shape[0], d), dtype=np.float64)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    _check("oscar_score_weighted_rows", lib.oscar_score_weighted_rows(
        q.ctypes.data, q.shape[0], k.ctypes.data, v.ctypes.data, k.shape[0], d, scale, out.ctypes.data))
    return out


def oscar_clip_threshold(acts: np.ndarray, r: np.ndarray, quantile: float = 0.999) -> float:
    """acts [n_heads][rows][d], r [n_heads][d][d] (host float64)."""
    acts, r = _f64(acts), _f64(r)
    h, rows, d = acts.shape
    tau = c_double(0.0)
    _check("oscar_clip_threshold", lib.oscar_clip_threshold(
        acts.ctypes.data, rows, h, d, r.ctypes.data, quantile, ctypes.byref(tau)))
    return tau.value


def oscar_rotation_file_write(path: str, r_k: np.ndarray, r_v: np.ndarray, tau_k, tau_v) -> None:
    """r_k, r_v [n_layers][n_kv][d][d], tau_k, tau_v [n_layers] (stored as float32)."""
    r_k = np.ascontiguousarray(r_k, dtype=np.float32)
    r_v = np.ascontiguousarray(r_v, dtype=np.float32)
    tk = np.ascontiguousarray(np.atleast_1d(tau_k), dtype=np.float32)
    tv = np.ascontiguousarray(np.atleast_1d(tau_v), dtype=np.float32)
    n_layers, n_kv, d = r_k.shape[0], r_k.shape[1], r_k.shape[2]
    _check("oscar_rotation_file_write", lib.oscar_rotation_file_write(
        os.fsencode(path), n_layers, n_kv, d, r_k.ctypes.data, r_v.ctypes.data, tk.ctypes.data, tv.ctypes.data))


def oscar_rotation_file_read(path: str):
    """(r_k, r_v [n_layers][n_kv][d][d] float32, tau_k, tau_v [n_layers] float32)."""
    dims = [c_int32(0), c_int32(0), c_int32(0)]
    _check("oscar_rotation_file_info", lib.oscar_rotation_file_info(os.fsencode(path), *[ctypes.byref(x) for x in dims]))
    n_layers, n_kv, d = (x.value for x in dims)
    r_k = np.empty((n_layers, n_kv, d, d), np.float32)
    r_v = np.empty_like(r_k)
    tk = np.empty(n_layers, np.float32)
    tv = np.empty(n_layers, np.float32)
    _check("oscar_rotation_file_read", lib.oscar_rotation_file_read(
        os.fsencode(path), n_layers, n_kv, d, r_k.ctypes.data, r_v.ctypes.data, tk.ctypes.data, tv.ctypes.data))
    return r_k, r_v, tk, tv


def oscar_fit_codebook(x: np.ndarray, r: np.ndarray, tau: float, iters: int = 100) -> np.ndarray:
    """Four Lloyd-Max levels (float32 holding fp16 values) from calibration rows
    x [n][d] rotated by r [d][d] and clipped at tau (host float64)."""
    x, r = _f64(x), _f64(r)
    out = np.empty(4, dtype=np.float32)
    _check("oscar_fit_codebook", lib.oscar_fit_codebook(x.ctypes.data, x.shape[0], x.shape[1], r.ctypes.data,
                                                        float(tau), int(iters), out.ctypes.data))
    return out


def oscar_quantize_append(desc: LayerDesc, k_src, v_src, src_rows: int, row_stride: int, src_index,
                          dst_req, dst_pos, n: int, new_k=None, new_v=None, stream=None) -> None:
    _check("oscar_quantize_append", lib.oscar_quantize_append(
        ctypes.byref(desc), _ptr(k_src), _ptr(v_src), int(src_rows), int(row_stride), _ptr(src_index),
        _ptr(dst_req), _ptr(dst_pos), int(n), _ptr(new_k), _ptr(new_v), _stream(stream)))


def oscar_quantize_append_overlapped(desc: LayerDesc, k_src, v_src, src_rows: int, row_stride: int, src_index,
                                     dst_req, dst_pos, n: int, new_k=None, new_v=None, stream=None) -> None:
    _check("oscar_quantize_append_overlapped", lib.oscar_quantize_append_overlapped(
        ctypes.byref(desc), _ptr(k_src), _ptr(v_src), int(src_rows), int(row_stride), _ptr(src_index),
        _ptr(dst_req), _ptr(dst_pos), int(n), _ptr(new_k), _ptr(new_v), _stream(stream)))


def oscar_decode_workspace_bytes(desc: LayerDesc) -> int:
    size = c_size_t(0)
    _check("oscar_decode_attention", lib.oscar_decode_attention(
        ctypes.byref(desc), None, None, None, ctypes.byref(size), None))
    return size.value


def oscar_decode_attention(desc: LayerDesc, q, out, workspace, workspace_bytes: int = None,
                           stream=None) -> None:
    size = c_size_t(workspace.numel() * workspace.element_size() if workspace_bytes is None
                    else workspace_bytes)
    _check("oscar_decode_attention", lib.oscar_decode_attention(
        ctypes.byref(desc), _ptr(q), _ptr(out), _ptr(workspace), ctypes.byref(size), _stream(stream)))


def oscar_decode_step(desc: LayerDesc, host_in, dev_in, in_bytes: int, k_src, v_src, src_rows: int,
                      row_stride: int, src_index, dst_req, dst_pos, n: int, new_k, new_v, q, out, workspace,
                      workspace_bytes: int, host_out=None, stream=None, flags: int = 0) -> None:
    """One decode step: H2D copy of the staged inputs, demotion, decode, D2H copy of the output.
    flags: 0 or OSCAR_STEP_OVERLAP_PREVIOUS (the demotion overlaps the kernel before it)."""
    _check("oscar_decode_step", lib.oscar_decode_step(
        ctypes.byref(desc), _ptr(host_in), _ptr(dev_in), int(in_bytes), _ptr(k_src), _ptr(v_src), int(src_rows),
        int(row_stride), _ptr(src_index), _ptr(dst_req), _ptr(dst_pos), int(n), _ptr(new_k), _ptr(new_v),
        _ptr(q), _ptr(out), _ptr(workspace), int(workspace_bytes), _ptr(host_out), int(flags), _stream(stream)))


def oscar_decode_attention_static(desc: LayerDesc, q, out, stream=None) -> None:
    """Decode attention with the library's fixed workspace (no allocation by anyone)."""
    _check("oscar_decode_attention_static", lib.oscar_decode_attention_static(
        ctypes.byref(desc), _ptr(q), _ptr(out), _stream(stream)))
