"""ctypes binding of liboscar.so (include/oscar.h).  Argument marshalling only:
every step of the path runs in the library.  The functions keep the C names.

Device arguments are torch CUDA tensors (PyTorch is used for device memory and
streams); host-side calls take numpy arrays.  A missing library raises at
import time -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "liboscar.so")

OSCAR_OK = 0
STATUS_NAMES = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "WORKSPACE", -4: "CUDA",
                -5: "NOT_CONVERGED"}
DEVERR_PAGE_ID, DEVERR_TIMEOUT, DEVERR_SEQ_LEN, DEVERR_NONFINITE = 1, 2, 4, 8
VARIANT_OSCAR, VARIANT_HADAMARD, VARIANT_IDENTITY = 0, 1, 2
EXPORTED = ("oscar_query_covariance", "oscar_score_covariance", "oscar_build_rotation",
            "oscar_prefill_quantize", "oscar_quantize_append", "oscar_decode_workspace_size",
            "oscar_decode_attention", "oscar_decode_attention_bf16", "oscar_device_sm_count",
            "oscar_status_string", "oscar_version", "oscar_decode_attention_static",
            "oscar_decode_step", "oscar_decode_step_rope", "oscar_multiquery_attention",
            "oscar_multiquery_workspace_size", "oscar_decode_step_host_staging_size",
            "oscar_decode_step_host",
            "oscar_calibration_workspace_size", "oscar_query_covariance_device",
            "oscar_score_covariance_device", "oscar_clip_threshold_device",
            "oscar_prefill_quantize_trace", "oscar_quantize_append_trace")


class OscarError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status} ({STATUS_NAMES.get(status, '?')}: "
                         f"{lib().oscar_status_string(status).decode()})")


class CacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("sink", ctypes.c_int32), ("window", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("num_int2_pages", ctypes.c_int64), ("num_bf16_pages", ctypes.c_int64),
        ("int2_pool", ctypes.c_void_p), ("bf16_pool", ctypes.c_void_p),
        ("int2_page_table", ctypes.c_void_p), ("bf16_page_table", ctypes.c_void_p),
        ("r_k", ctypes.c_void_p), ("r_v", ctypes.c_void_p),
        ("clip_k", ctypes.c_void_p), ("clip_v", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("code_bits", ctypes.c_int32),
    ]


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m int2_rotated_kv_gb300.build` (no fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        sig = {
            "oscar_query_covariance": (I32, [I32, I32, I64, P, P]),
            "oscar_score_covariance": (I32, [I32, I32, I64, P, P, P, I32, P]),
            "oscar_build_rotation": (I32, [I32, P, P, I64, D, I32, P, P, P, P]),
            "oscar_prefill_quantize": (I32, [P, P, P, P, P, P, I32, I64, P]),
            "oscar_quantize_append": (I32, [P, P, P, P, I32, P]),
            "oscar_prefill_quantize_trace": (I32, [P, P, P, P, P, P, I32, I64, P, P]),
            "oscar_quantize_append_trace": (I32, [P, P, P, P, I32, P, P]),
            "oscar_decode_workspace_size": (ctypes.c_size_t, [P, I32, I32]),
            "oscar_multiquery_workspace_size": (ctypes.c_size_t, [P, I32, I32, I32]),
            "oscar_decode_attention": (I32, [P, P, P, I32, I32, P, P, ctypes.c_size_t, P]),
            "oscar_decode_attention_bf16": (I32, [P, P, P, I32, I32, P, P, ctypes.c_size_t, P]),
            "oscar_device_sm_count": (I32, []),
            "oscar_decode_attention_static": (I32, [P, P, P, I32, I32, P, P]),
            "oscar_decode_step": (I32, [P, P, P, P, P, I32, I32, P, P, ctypes.c_size_t, P]),
            "oscar_decode_step_rope": (I32, [P, P, P, P, P, I32, I32, D, P, P, ctypes.c_size_t, P]),
            "oscar_decode_step_host_staging_size": (ctypes.c_size_t, [P, I32]),
            "oscar_decode_step_host": (I32, [P, P, P, I32, I32, D, P, P, ctypes.c_size_t, P,
                                             ctypes.c_size_t, P]),
            "oscar_multiquery_attention": (I32, [P, P, P, P, I32, I32, I32, P, P, ctypes.c_size_t, P]),
            "oscar_calibration_workspace_size": (ctypes.c_size_t, [I32, I32, I32, I64]),
            "oscar_query_covariance_device": (I32, [I32, I32, I32, I64, P, P, P, ctypes.c_size_t, P]),
            "oscar_score_covariance_device": (I32, [I32, I32, I32, I64, P, P, P, P, P,
                                                    ctypes.c_size_t, P]),
            "oscar_clip_threshold_device": (I32, [I32, I32, I64, P, P, D, P, P, ctypes.c_size_t, P]),
            "oscar_status_string": (ctypes.c_char_p, [I32]),
            "oscar_version": (I32, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(fn: str, status: int) -> None:
    if status != OSCAR_OK:
        raise OscarError(fn, status)


def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ host calls

def oscar_query_covariance(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float32)
    n, g, d = q.shape
    c = np.zeros((d, d), np.float64)
    _check("oscar_query_covariance", lib().oscar_query_covariance(d, g, n, _np_ptr(q), _np_ptr(c)))
    return c


def oscar_score_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray, num_threads: int = 0):
    q = np.ascontiguousarray(q, np.float32)
    k = np.ascontiguousarray(k, np.float32)
    v = np.ascontiguousarray(v, np.float32)
    n, g, d = q.shape
    c = np.zeros((d, d), np.float64)
    _check("oscar_score_covariance",
           lib().oscar_score_covariance(d, g, n, _np_ptr(q), _np_ptr(k), _np_ptr(v), num_threads,
                                        _np_ptr(c)))
    return c


def oscar_build_rotation(c, calib_x: np.ndarray, percentile: float = 99.9,
                         variant: int = VARIANT_OSCAR):
    """Returns (R64 [d,d] fp64, R32 [d,d] fp32, clip float32, eigenvalues [d])."""
    x = np.ascontiguousarray(calib_x, np.float32)
    n, d = x.shape
    cc = None if c is None else np.ascontiguousarray(c, np.float64)
    r64 = np.zeros((d, d), np.float64)
    r32 = np.zeros((d, d), np.float32)
    clip = np.zeros(1, np.float32)
    ev = np.zeros(d, np.float64)
    _check("oscar_build_rotation",
           lib().oscar_build_rotation(d, None if cc is None else _np_ptr(cc), _np_ptr(x), n,
                                      float(percentile), variant, _np_ptr(r64), _np_ptr(r32),
                                      _np_ptr(clip), _np_ptr(ev)))
    return r64, r32, np.float32(clip[0]), ev


# --------------------------------------------------------------- device calls

def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


@dataclasses.dataclass
class Cache:
    """Device tensors of one layer's cache plus its C descriptor.

    int2_pool: uint8 [num_int2_pages * Hkv * 12d] (INT4 variant, code_bits 4:
    20d per page-head); bf16_pool: bfloat16 [num_bf16_pages * Hkv * 32d]; page
    tables int32 [batch, max_pages_per_seq]; r_k, r_v fp32 [Hkv, d, d]; clip_k,
    clip_v fp32 [Hkv]; status int32 [1].
    """
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    sink: int
    window: int
    int2_pool: object
    bf16_pool: object
    int2_page_table: object
    bf16_page_table: object
    r_k: object = None
    r_v: object = None
    clip_k: object = None
    clip_v: object = None
    status: object = None
    code_bits: int = 2

    def desc(self) -> CacheDesc:
        key = tuple(_ptr(t) for t in (self.int2_pool, self.bf16_pool, self.int2_page_table,
                                      self.bf16_page_table, self.r_k, self.r_v, self.clip_k,
                                      self.clip_v, self.status)) + (self.code_bits,)
        cached = self.__dict__.get("_desc")
        if cached is not None and cached[0] == key:
            return cached[1]
        d = self.head_dim
        desc = CacheDesc(
            self.num_kv_heads, self.num_q_heads, d, self.sink, self.window,
            int(self.bf16_page_table.shape[1]),
            0 if self.int2_pool is None
            else self.int2_pool.numel() // (self.num_kv_heads * (4 * self.code_bits + 4) * d),
            self.bf16_pool.numel() // (self.num_kv_heads * 32 * d),
            _ptr(self.int2_pool), _ptr(self.bf16_pool), _ptr(self.int2_page_table),
            _ptr(self.bf16_page_table), _ptr(self.r_k), _ptr(self.r_v), _ptr(self.clip_k),
            _ptr(self.clip_v), _ptr(self.status), self.code_bits)
        self.__dict__["_desc"] = (key, desc)
        return desc


def oscar_prefill_quantize(cache: Cache, k, v, seq_ids, positions, seq_lens_final, stream=None):
    d = cache.desc()
    _check("oscar_prefill_quantize",
           lib().oscar_prefill_quantize(ctypes.byref(d), _ptr(k), _ptr(v), _ptr(seq_ids),
                                        _ptr(positions), _ptr(seq_lens_final),
                                        int(seq_lens_final.numel()), int(seq_ids.numel()),
                                        _stream(stream)))


def oscar_quantize_append(cache: Cache, k_new, v_new, seq_lens_after, stream=None):
    d = cache.desc()
    _check("oscar_quantize_append",
           lib().oscar_quantize_append(ctypes.byref(d), _ptr(k_new), _ptr(v_new),
                                       _ptr(seq_lens_after), int(seq_lens_after.numel()),
                                       _stream(stream)))


def oscar_prefill_quantize_trace(cache: Cache, k, v, seq_ids, positions, seq_lens_final, y_out,
                                 stream=None):
    """oscar_prefill_quantize that also writes the fp32 rotated values of every
    INT2 placement to y_out (float32 [total_tokens, Hkv, 2, d], device)."""
    d = cache.desc()
    _check("oscar_prefill_quantize_trace",
           lib().oscar_prefill_quantize_trace(ctypes.byref(d), _ptr(k), _ptr(v), _ptr(seq_ids),
                                              _ptr(positions), _ptr(seq_lens_final),
                                              int(seq_lens_final.numel()), int(seq_ids.numel()),
                                              _ptr(y_out), _stream(stream)))


def oscar_quantize_append_trace(cache: Cache, k_new, v_new, seq_lens_after, y_out, stream=None):
    """oscar_quantize_append that also writes the fp32 rotated values of each
    token leaving the window to y_out (float32 [batch, Hkv, 2, d], device)."""
    d = cache.desc()
    _check("oscar_quantize_append_trace",
           lib().oscar_quantize_append_trace(ctypes.byref(d), _ptr(k_new), _ptr(v_new),
                                             _ptr(seq_lens_after), int(seq_lens_after.numel()),
                                             _ptr(y_out), _stream(stream)))


def oscar_decode_workspace_size(cache: Cache, batch: int, max_seq_len: int) -> int:
    d = cache.desc()
    return int(lib().oscar_decode_workspace_size(ctypes.byref(d), batch, max_seq_len))


def oscar_multiquery_workspace_size(cache: Cache, batch: int, m_rows: int, max_seq_len: int) -> int:
    d = cache.desc()
    return int(lib().oscar_multiquery_workspace_size(ctypes.byref(d), batch, m_rows, max_seq_len))


def oscar_decode_attention(cache: Cache, q, seq_lens, max_seq_len: int, out, workspace,
                           stream=None):
    d = cache.desc()
    _check("oscar_decode_attention",
           lib().oscar_decode_attention(ctypes.byref(d), _ptr(q), _ptr(seq_lens),
                                        int(seq_lens.numel()), int(max_seq_len), _ptr(out),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))


def oscar_decode_attention_bf16(cache: Cache, q, seq_lens, max_seq_len: int, out, workspace,
                                stream=None):
    d = cache.desc()
    _check("oscar_decode_attention_bf16",
           lib().oscar_decode_attention_bf16(ctypes.byref(d), _ptr(q), _ptr(seq_lens),
                                             int(seq_lens.numel()), int(max_seq_len), _ptr(out),
                                             _ptr(workspace),
                                             workspace.numel() * workspace.element_size(),
                                             _stream(stream)))


def oscar_decode_step(cache: Cache, q, k_new, v_new, seq_lens_after, max_seq_len: int, out,
                      workspace, stream=None):
    """Append the step's new token (and move the one leaving the window to INT2),
    then attend at the new lengths: one fused call, same result as
    oscar_quantize_append followed by oscar_decode_attention."""
    d = cache.desc()
    _check("oscar_decode_step",
           lib().oscar_decode_step(ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new),
                                   _ptr(seq_lens_after), int(seq_lens_after.numel()),
                                   int(max_seq_len), _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def oscar_decode_step_rope(cache: Cache, q, k_new, v_new, seq_lens_after, max_seq_len: int,
                           rope_base: float, out, workspace, stream=None):
    """The fused decode step with the rotary embedding of the new query and key."""
    d = cache.desc()
    _check("oscar_decode_step_rope",
           lib().oscar_decode_step_rope(ctypes.byref(d), _ptr(q), _ptr(k_new), _ptr(v_new),
                                        _ptr(seq_lens_after), int(seq_lens_after.numel()),
                                        int(max_seq_len), float(rope_base), _ptr(out),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)))


def oscar_decode_step_host_staging_size(cache: Cache, batch: int) -> int:
    """Device staging bytes of oscar_decode_step_host for `batch` sequences."""
    return int(lib().oscar_decode_step_host_staging_size(ctypes.byref(cache.desc()), int(batch)))


def oscar_decode_step_host(cache: Cache, in_host, seq_lens_after, max_seq_len: int, out_host,
                           staging, workspace, rope_base: float = 0.0, stream=None):
    """The fused decode step with its inputs and result in host memory.

    in_host: host bf16 tensor holding q [B][Hq][d], k_new [B][Hkv][d] and
    v_new [B][Hkv][d] back to back (pinned for asynchronous copies); out_host:
    host bf16 [B][Hq][d]; staging, workspace: device bytes.  Everything is
    queued on the stream; synchronise it before reading out_host."""
    d = cache.desc()
    _check("oscar_decode_step_host",
           lib().oscar_decode_step_host(ctypes.byref(d), _ptr(in_host), _ptr(seq_lens_after),
                                        int(seq_lens_after.numel()), int(max_seq_len),
                                        float(rope_base), _ptr(out_host), _ptr(staging),
                                        staging.numel() * staging.element_size(), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)))


def oscar_multiquery_attention(cache: Cache, q, seq_lens, q_pos, max_seq_len: int, out, workspace,
                               stream=None):
    """Several query rows per sequence (q [B][M][Hq][d], q_pos [B][M]) over the
    mixed cache; row (b, m) attends to stored tokens 0 .. q_pos[b][m]."""
    d = cache.desc()
    B, M = int(q_pos.shape[0]), int(q_pos.shape[1])
    _check("oscar_multiquery_attention",
           lib().oscar_multiquery_attention(ctypes.byref(d), _ptr(q), _ptr(seq_lens), _ptr(q_pos),
                                            B, M, int(max_seq_len), _ptr(out), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream)))


def oscar_decode_attention_static(cache: Cache, q, seq_lens, max_seq_len: int, out, stream=None):
    """Decode attention without a workspace argument, for callers that cannot
    allocate device memory: the library's own fixed 16 MiB scratch buffer is
    used and nothing is allocated.  Calls must not overlap on the GPU."""
    d = cache.desc()
    _check("oscar_decode_attention_static",
           lib().oscar_decode_attention_static(ctypes.byref(d), _ptr(q), _ptr(seq_lens),
                                               int(seq_lens.numel()), int(max_seq_len), _ptr(out),
                                               _stream(stream)))


def oscar_calibration_workspace_size(num_kv_heads: int, num_q_heads: int, d: int, n: int) -> int:
    return int(lib().oscar_calibration_workspace_size(num_kv_heads, num_q_heads, d, n))


def _ws_bytes(workspace) -> int:
    return workspace.numel() * workspace.element_size()


def oscar_query_covariance_device(q, num_kv_heads: int, c_out, workspace, stream=None):
    """C_Q per KV head on the device: q bf16 [n][Hq][d] -> c_out fp64 [Hkv][d][d]."""
    n, hq, d = (int(x) for x in q.shape)
    _check("oscar_query_covariance_device",
           lib().oscar_query_covariance_device(num_kv_heads, hq, d, n, _ptr(q), _ptr(c_out),
                                               _ptr(workspace), _ws_bytes(workspace),
                                               _stream(stream)))


def oscar_score_covariance_device(q, k, v, c_out, workspace, stream=None):
    """C_S per KV head on the device: q bf16 [n][Hq][d], k/v bf16 [n][Hkv][d]."""
    n, hq, d = (int(x) for x in q.shape)
    hkv = int(k.shape[1])
    _check("oscar_score_covariance_device",
           lib().oscar_score_covariance_device(hkv, hq, d, n, _ptr(q), _ptr(k), _ptr(v),
                                               _ptr(c_out), _ptr(workspace), _ws_bytes(workspace),
                                               _stream(stream)))


def oscar_clip_threshold_device(x, r, percentile: float, clip_out, workspace, stream=None):
    """Clip per KV head on the device: x bf16 [n][Hkv][d], r fp32 [Hkv][d][d]."""
    n, hkv, d = (int(x_) for x_ in x.shape)
    _check("oscar_clip_threshold_device",
           lib().oscar_clip_threshold_device(hkv, d, n, _ptr(x), _ptr(r), float(percentile),
                                             _ptr(clip_out), _ptr(workspace), _ws_bytes(workspace),
                                             _stream(stream)))


def oscar_device_sm_count() -> int:
    return int(lib().oscar_device_sm_count())


def oscar_version() -> int:
    return int(lib().oscar_version())
