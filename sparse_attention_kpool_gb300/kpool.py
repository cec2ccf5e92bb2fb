"""ctypes binding of the CUDA library (C ABI in include/kpool.h).

Argument marshalling only: every step of the selection runs in the library's
kernels. Functions carry the C names. Tensors must be CUDA tensors on the
current device; outputs and workspace are allocated with torch when the caller
does not pass them (the library itself never allocates). Calls run on torch's
current CUDA stream unless `stream` is given.

There is no fallback: if the library is not built, or a call fails, these
functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkpool.so")

KPOOL_OK = 0
KPOOL_ERR_INVALID_ARG = 1
KPOOL_ERR_UNSUPPORTED = 2
KPOOL_ERR_WORKSPACE = 3
KPOOL_ERR_CUDA = 4
KPOOL_ERR_DEVICE_TIMEOUT = 5
KPOOL_ERR_INTERNAL = 6

KPOOL_BF16 = 0
KPOOL_F32 = 1

KPOOL_SCORE_AUTO = 0
KPOOL_SCORE_TC = 1
KPOOL_SCORE_SIMT = 2

EXPORTED = (
    "kpool_workspace_bytes", "kpool_select", "kpool_select_ex", "kpool_pool_keys", "kpool_expand",
    "kpool_last_device_error", "kpool_wait_timeout_selftest", "kpool_status_string", "kpool_last_cuda_error",
    "kpool_select_static_scratch", "kpool_rows_workspace_bytes", "kpool_select_rows", "kpool_select_rows_ex",
    "kpool_pool_keys_gated", "kpool_select_pooled", "kpool_static_scratch_last_device_error",
    "kpool_balanced_row_split", "kpool_index_scores", "kpool_index_scores_pooled",
)
KPOOL_STATIC_SCRATCH_BYTES = 48 << 20


class KpoolError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = f" [{kpool_last_cuda_error()}]" if status == KPOOL_ERR_CUDA else ""
        super().__init__(f"{what}: {kpool_status_string(status)} (status {status}){detail}")


KPOOL_OPT_ROW_RANGE = 1


class kpool_options(ctypes.Structure):
    _fields_ = [("score_kernel", ctypes.c_int32), ("max_ctas", ctypes.c_int32),
                ("stage_events", ctypes.POINTER(ctypes.c_void_p)), ("row_begin", ctypes.c_int32),
                ("row_end", ctypes.c_int32), ("flags", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Open the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"the KPool CUDA library is not built ({LIB_PATH} missing); "
                               "run `python -m sparse_attention_kpool_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        lib.kpool_workspace_bytes.argtypes = [i64, i32, i32, i32, i32, i32, i32]
        lib.kpool_workspace_bytes.restype = sz
        sel = [P, P, P, P, i32, i64, i32, i32, i32, i32, i32, f32, P, P, P, P, sz, P]
        lib.kpool_select.argtypes = sel
        lib.kpool_select.restype = i32
        lib.kpool_select_ex.argtypes = sel + [ctypes.POINTER(kpool_options)]
        lib.kpool_select_ex.restype = i32
        lib.kpool_pool_keys.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, sz, P]
        lib.kpool_pool_keys.restype = i32
        lib.kpool_expand.argtypes = [P, P, i32, i64, i32, i32, P, P]
        lib.kpool_expand.restype = i32
        lib.kpool_last_device_error.argtypes = [P, P]
        lib.kpool_last_device_error.restype = i32
        lib.kpool_wait_timeout_selftest.argtypes = [P, sz, i64, P]
        lib.kpool_wait_timeout_selftest.restype = i32
        lib.kpool_status_string.argtypes = [i32]
        lib.kpool_status_string.restype = ctypes.c_char_p
        lib.kpool_last_cuda_error.argtypes = []
        lib.kpool_last_cuda_error.restype = ctypes.c_char_p
        lib.kpool_select_static_scratch.argtypes = [P, P, P, P, i32, i64, i32, i32, i32, i32, i32, f32, P, P, P, P]
        lib.kpool_select_static_scratch.restype = i32
        lib.kpool_static_scratch_last_device_error.argtypes = [P]
        lib.kpool_static_scratch_last_device_error.restype = i32
        lib.kpool_rows_workspace_bytes.argtypes = [i32, i64, i32, i32, i32]
        lib.kpool_rows_workspace_bytes.restype = sz
        lib.kpool_select_rows.argtypes = [P, P, P, P, i32, P, P, i32, i64, i32, i32, i32, i32, i32, f32, P, P, P,
                                          P, sz, P]
        lib.kpool_select_rows.restype = i32
        lib.kpool_select_rows_ex.argtypes = lib.kpool_select_rows.argtypes + [ctypes.POINTER(kpool_options)]
        lib.kpool_select_rows_ex.restype = i32
        lib.kpool_pool_keys_gated.argtypes = [P, P, P, P, i32, i64, i32, i32, i32, P, P, sz, P]
        lib.kpool_pool_keys_gated.restype = i32
        lib.kpool_select_pooled.argtypes = sel + [ctypes.POINTER(kpool_options)]
        lib.kpool_select_pooled.restype = i32
        lib.kpool_balanced_row_split.argtypes = [P, i32, i32, i64, i32, P]
        lib.kpool_balanced_row_split.restype = i32
        isc = [P, P, P, P, i32, i64, i32, i32, i32, i32, f32, P, i64, P, sz, P, ctypes.POINTER(kpool_options)]
        lib.kpool_index_scores.argtypes = isc
        lib.kpool_index_scores.restype = i32
        lib.kpool_index_scores_pooled.argtypes = isc
        lib.kpool_index_scores_pooled.restype = i32
        _lib = lib
        return lib


def kpool_status_string(status: int) -> str:
    return load().kpool_status_string(int(status)).decode()


def kpool_last_cuda_error() -> str:
    return load().kpool_last_cuda_error().decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KPOOL_BF16
    if t.dtype == torch.float32:
        return KPOOL_F32
    raise TypeError(f"q/k must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def kpool_workspace_bytes(total_tokens: int, num_seqs: int, heads: int, head_dim: int, dtype: int, kpool: int,
                          index_topk: int) -> int:
    return int(load().kpool_workspace_bytes(total_tokens, num_seqs, heads, head_dim, dtype, kpool, index_topk))


def new_workspace(total_tokens: int, num_seqs: int, heads: int, head_dim: int, dtype: int, kpool: int,
                  index_topk: int, device=None) -> torch.Tensor:
    n = kpool_workspace_bytes(total_tokens, num_seqs, heads, head_dim, dtype, kpool, index_topk)
    if n == 0:
        raise KpoolError(KPOOL_ERR_INVALID_ARG, "kpool_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def kpool_select_ex(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, cu_seqlens: torch.Tensor, kpool: int,
                    index_topk: int, scale: float, out_pool_ids=None, out_token_ids=None, out_pool_scores=None,
                    return_scores: bool = False, workspace=None, stream=None, score_kernel: int = KPOOL_SCORE_AUTO,
                    max_ctas: int = 0, stage_events=None, row_range=None):
    """q [T,H,d], k [T,d] (bf16 or fp32), w [T,H] fp32, cu_seqlens [S+1] int32 -> (pool_ids [R,B],
    token_ids [R, index_topk+kpool], pool_scores [R,B] or None), R = T rows, or the rows of
    row_range = (row_begin, row_end) (a shard of query rows; no scores on that path).

    stage_events: optional 5 already-recorded torch.cuda.Event(enable_timing=True); the library
    re-records them around its four kernels (see kpool_options in kpool.h)."""
    T, H, d = q.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if k.dtype != q.dtype or w.dtype != torch.float32 or cu_seqlens.dtype != torch.int32:
        raise TypeError("k must match q's dtype; w must be float32; cu_seqlens int32")
    B = index_topk // kpool if kpool > 0 else 0
    R = T if row_range is None else max(0, int(row_range[1]) - int(row_range[0]))
    dev = q.device
    if out_pool_ids is None:
        out_pool_ids = torch.empty((R, B), dtype=torch.int32, device=dev)
    if out_token_ids is None:
        out_token_ids = torch.empty((R, index_topk + kpool), dtype=torch.int32, device=dev)
    if out_pool_scores is None and return_scores:
        out_pool_scores = torch.empty((R, B), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, S, H, d, dt, kpool, index_topk, dev)
    _check_cuda(q, k, w, cu_seqlens, out_pool_ids, out_token_ids, out_pool_scores, workspace)
    opts, _arr = _options(score_kernel, max_ctas, row_range, stage_events)
    st = load().kpool_select_ex(_ptr(q), _ptr(k), _ptr(w), _ptr(cu_seqlens), S, T, H, d, dt, kpool, index_topk,
                                float(scale), _ptr(out_pool_ids), _ptr(out_token_ids), _ptr(out_pool_scores),
                                _ptr(workspace), workspace.numel(), _stream(stream), ctypes.byref(opts))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_select")
    return out_pool_ids, out_token_ids, out_pool_scores


def kpool_select(q, k, w, cu_seqlens, kpool, index_topk, scale, out_pool_ids=None, out_token_ids=None,
                 out_pool_scores=None, return_scores=False, workspace=None, stream=None):
    """The whole selection with default options (see kpool_select_ex)."""
    return kpool_select_ex(q, k, w, cu_seqlens, kpool, index_topk, scale, out_pool_ids, out_token_ids,
                           out_pool_scores, return_scores, workspace, stream)


def kpool_pool_keys(k: torch.Tensor, cu_seqlens: torch.Tensor, kpool: int, out=None, workspace=None, stream=None):
    """Mean-pooled keys; returns a [T // kpool, d] tensor whose first P rows are the pools."""
    T, d = k.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(k)
    if out is None:
        out = torch.empty((max(T // kpool, 0), d), dtype=k.dtype, device=k.device)
    if workspace is None:
        workspace = new_workspace(T, S, 1, d, dt, kpool, 0, k.device)
    _check_cuda(k, cu_seqlens, out, workspace)
    st = load().kpool_pool_keys(_ptr(k), _ptr(cu_seqlens), S, T, d, dt, kpool, _ptr(out), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_pool_keys")
    return out


def kpool_expand(pool_ids: torch.Tensor, cu_seqlens: torch.Tensor, kpool: int, index_topk: int, out=None,
                 stream=None):
    T = pool_ids.shape[0]
    S = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, index_topk + kpool), dtype=torch.int32, device=pool_ids.device)
    _check_cuda(pool_ids, cu_seqlens, out)
    st = load().kpool_expand(_ptr(pool_ids), _ptr(cu_seqlens), S, T, kpool, index_topk, _ptr(out), _stream(stream))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_expand")
    return out


def kpool_last_device_error(workspace: torch.Tensor, stream=None) -> int:
    return int(load().kpool_last_device_error(_ptr(workspace), _stream(stream)))


def kpool_wait_timeout_selftest(workspace: torch.Tensor, spin_limit: int, stream=None) -> int:
    return int(load().kpool_wait_timeout_selftest(_ptr(workspace), workspace.numel(), int(spin_limit),
                                                  _stream(stream)))


def kpool_select_static_scratch(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, cu_seqlens: torch.Tensor,
                                kpool: int, index_topk: int, scale: float, out_pool_ids=None, out_token_ids=None,
                                out_pool_scores=None, return_scores: bool = False, stream=None):
    """kpool_select with the library's built-in scratch array instead of a workspace (for callers
    that cannot allocate device memory; see kpool_select_static_scratch in kpool.h). The outputs
    are allocated here only when not passed."""
    T, H, d = q.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    B = index_topk // kpool if kpool > 0 else 0
    dev = q.device
    if out_pool_ids is None:
        out_pool_ids = torch.empty((T, B), dtype=torch.int32, device=dev)
    if out_token_ids is None:
        out_token_ids = torch.empty((T, index_topk + kpool), dtype=torch.int32, device=dev)
    if out_pool_scores is None and return_scores:
        out_pool_scores = torch.empty((T, B), dtype=torch.float32, device=dev)
    _check_cuda(q, k, w, cu_seqlens, out_pool_ids, out_token_ids, out_pool_scores)
    st = load().kpool_select_static_scratch(_ptr(q), _ptr(k), _ptr(w), _ptr(cu_seqlens), S, T, H, d, dt, kpool,
                                            index_topk, float(scale), _ptr(out_pool_ids), _ptr(out_token_ids),
                                            _ptr(out_pool_scores), _stream(stream))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_select_static_scratch")
    return out_pool_ids, out_token_ids, out_pool_scores


def kpool_static_scratch_last_device_error(stream=None) -> int:
    """Device error word of the last kpool_select_static_scratch call on this device (syncs)."""
    return int(load().kpool_static_scratch_last_device_error(_stream(stream)))


def kpool_rows_workspace_bytes(num_rows: int, total_tokens: int, num_seqs: int, kpool: int, index_topk: int) -> int:
    return int(load().kpool_rows_workspace_bytes(num_rows, total_tokens, num_seqs, kpool, index_topk))


def new_rows_workspace(num_rows: int, total_tokens: int, num_seqs: int, kpool: int, index_topk: int,
                       device=None) -> torch.Tensor:
    n = kpool_rows_workspace_bytes(num_rows, total_tokens, num_seqs, kpool, index_topk)
    if n == 0:
        raise KpoolError(KPOOL_ERR_INVALID_ARG, "kpool_rows_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def kpool_select_rows(q: torch.Tensor, w: torch.Tensor, row_seq: torch.Tensor, row_pos: torch.Tensor,
                      pooled_keys: torch.Tensor, cu_seqlens: torch.Tensor, total_tokens: int, kpool: int,
                      index_topk: int, scale: float, out_pool_ids=None, out_token_ids=None, out_pool_scores=None,
                      return_scores: bool = False, workspace=None, stream=None, max_ctas: int = 0,
                      stage_events=None):
    """Selection for explicit query rows against an existing pooled-key cache (decode).

    q [R,H,d] bf16, w [R,H] fp32, row_seq / row_pos [R] int32 (sequence and local position of
    each row), pooled_keys [>= P, d] as kpool_pool_keys returns them for cu_seqlens [S+1]
    (the key batch of total_tokens tokens) -> (pool_ids [R,B], token_ids [R, index_topk+kpool],
    pool_scores [R,B] or None).

    stage_events: optional 4 already-recorded timing events, re-recorded around the three kernels."""
    R, H, d = q.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if (pooled_keys.dtype != q.dtype or w.dtype != torch.float32 or cu_seqlens.dtype != torch.int32
            or row_seq.dtype != torch.int32 or row_pos.dtype != torch.int32):
        raise TypeError("pooled_keys must match q's dtype; w float32; cu_seqlens, row_seq, row_pos int32")
    B = index_topk // kpool if kpool > 0 else 0
    dev = q.device
    if out_pool_ids is None:
        out_pool_ids = torch.empty((R, B), dtype=torch.int32, device=dev)
    if out_token_ids is None:
        out_token_ids = torch.empty((R, index_topk + kpool), dtype=torch.int32, device=dev)
    if out_pool_scores is None and return_scores:
        out_pool_scores = torch.empty((R, B), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_rows_workspace(R, total_tokens, S, kpool, index_topk, dev)
    _check_cuda(q, w, row_seq, row_pos, pooled_keys, cu_seqlens, out_pool_ids, out_token_ids, out_pool_scores,
                workspace)
    opts = kpool_options(KPOOL_SCORE_AUTO, max_ctas)
    if stage_events is not None:
        if len(stage_events) != 4:
            raise ValueError("stage_events needs 4 events")
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(int(e.cuda_event)) for e in stage_events])
        if not all(arr):
            raise ValueError("record each event once before passing it (torch creates events lazily)")
        opts.stage_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    st = load().kpool_select_rows_ex(_ptr(q), _ptr(w), _ptr(row_seq), _ptr(row_pos), R, _ptr(pooled_keys),
                                     _ptr(cu_seqlens), S, int(total_tokens), H, d, dt, kpool, index_topk,
                                     float(scale), _ptr(out_pool_ids), _ptr(out_token_ids), _ptr(out_pool_scores),
                                     _ptr(workspace), workspace.numel(), _stream(stream), ctypes.byref(opts))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_select_rows")
    return out_pool_ids, out_token_ids, out_pool_scores


def kpool_pool_keys_gated(k: torch.Tensor, gate: torch.Tensor, ape: torch.Tensor, cu_seqlens: torch.Tensor,
                          kpool: int, out=None, workspace=None, stream=None):
    """Gated pooled keys (see kpool_pool_keys_gated in kpool.h): k [T,d], gate [T,d] fp32,
    ape [kpool,d] fp32 -> [T // kpool, d] whose first P rows are the pools."""
    T, d = k.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(k)
    if gate.dtype != torch.float32 or ape.dtype != torch.float32 or tuple(gate.shape) != (T, d) \
            or tuple(ape.shape) != (kpool, d):
        raise TypeError("gate must be float32 [T, d] and ape float32 [kpool, d]")
    if out is None:
        out = torch.empty((max(T // kpool, 0), d), dtype=k.dtype, device=k.device)
    if workspace is None:
        workspace = new_workspace(T, S, 1, d, dt, kpool, 0, k.device)
    _check_cuda(k, gate, ape, cu_seqlens, out, workspace)
    st = load().kpool_pool_keys_gated(_ptr(k), _ptr(gate), _ptr(ape), _ptr(cu_seqlens), S, T, d, dt, kpool, _ptr(out),
                                      _ptr(workspace), workspace.numel(), _stream(stream))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_pool_keys_gated")
    return out


def kpool_select_pooled(q: torch.Tensor, pooled_keys: torch.Tensor, w: torch.Tensor, cu_seqlens: torch.Tensor,
                        kpool: int, index_topk: int, scale: float, out_pool_ids=None, out_token_ids=None,
                        out_pool_scores=None, return_scores: bool = False, workspace=None, stream=None,
                        score_kernel: int = KPOOL_SCORE_AUTO, max_ctas: int = 0, row_range=None):
    """Selection from pooled keys the caller already has (steps 2-4); q [T,H,d], pooled_keys [>= P, d].
    row_range as for kpool_select_ex."""
    T, H, d = q.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if pooled_keys.dtype != q.dtype or w.dtype != torch.float32 or cu_seqlens.dtype != torch.int32:
        raise TypeError("pooled_keys must match q's dtype; w must be float32; cu_seqlens int32")
    B = index_topk // kpool if kpool > 0 else 0
    R = T if row_range is None else max(0, int(row_range[1]) - int(row_range[0]))
    dev = q.device
    if out_pool_ids is None:
        out_pool_ids = torch.empty((R, B), dtype=torch.int32, device=dev)
    if out_token_ids is None:
        out_token_ids = torch.empty((R, index_topk + kpool), dtype=torch.int32, device=dev)
    if out_pool_scores is None and return_scores:
        out_pool_scores = torch.empty((R, B), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, S, H, d, dt, kpool, index_topk, dev)
    _check_cuda(q, pooled_keys, w, cu_seqlens, out_pool_ids, out_token_ids, out_pool_scores, workspace)
    opts = kpool_options(score_kernel, max_ctas)
    if row_range is not None:
        opts.row_begin, opts.row_end = int(row_range[0]), int(row_range[1])
        opts.flags = KPOOL_OPT_ROW_RANGE
    st = load().kpool_select_pooled(_ptr(q), _ptr(pooled_keys), _ptr(w), _ptr(cu_seqlens), S, T, H, d, dt, kpool,
                                    index_topk, float(scale), _ptr(out_pool_ids), _ptr(out_token_ids),
                                    _ptr(out_pool_scores), _ptr(workspace), workspace.numel(), _stream(stream),
                                    ctypes.byref(opts))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_select_pooled")
    return out_pool_ids, out_token_ids, out_pool_scores


def _options(score_kernel, max_ctas, row_range, stage_events):
    """kpool_options for a call, plus the event array it points to (keep both alive)."""
    opts = kpool_options(score_kernel, max_ctas)
    if row_range is not None:
        opts.row_begin, opts.row_end = int(row_range[0]), int(row_range[1])
        opts.flags = KPOOL_OPT_ROW_RANGE
    arr = None
    if stage_events is not None:
        if len(stage_events) != 5:
            raise ValueError("stage_events needs 5 events")
        arr = (ctypes.c_void_p * 5)(*[ctypes.c_void_p(int(e.cuda_event)) for e in stage_events])
        if not all(arr):
            raise ValueError("record each event once before passing it (torch creates events lazily)")
        opts.stage_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    return opts, arr


def kpool_index_scores(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, cu_seqlens: torch.Tensor, kpool: int,
                       scale: float, ld: int | None = None, out=None, row_range=None, workspace=None, stream=None,
                       score_kernel: int = KPOOL_SCORE_AUTO, max_ctas: int = 0, stage_events=None,
                       pooled: bool = False):
    """Full index scores [R, ld] fp32 of the rows [row_begin, row_end) (all T rows without
    row_range): element (i, p) is the score of pool p of the row's sequence when the row may
    see it, else -inf. ld defaults to T // kpool. With pooled=True, `k` holds pooled keys
    (kpool_index_scores_pooled)."""
    T, H, d = q.shape
    S = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if k.dtype != q.dtype or w.dtype != torch.float32 or cu_seqlens.dtype != torch.int32:
        raise TypeError("k must match q's dtype; w must be float32; cu_seqlens int32")
    if ld is None:
        ld = max(1, T // kpool) if kpool > 0 else 1
    R = T if row_range is None else max(0, int(row_range[1]) - int(row_range[0]))
    dev = q.device
    if out is None:
        out = torch.empty((R, ld), dtype=torch.float32, device=dev)
    elif out.dtype != torch.float32 or out.numel() < R * ld or not out.is_contiguous():
        raise TypeError("out must be a contiguous float32 tensor of at least R * ld elements")
    if workspace is None:
        workspace = new_workspace(T, S, H, d, dt, kpool, 0, dev)
    _check_cuda(q, k, w, cu_seqlens, out, workspace)
    opts, _arr = _options(score_kernel, max_ctas, row_range, stage_events)
    fn = load().kpool_index_scores_pooled if pooled else load().kpool_index_scores
    st = fn(_ptr(q), _ptr(k), _ptr(w), _ptr(cu_seqlens), S, T, H, d, dt, kpool, float(scale), _ptr(out), int(ld),
            _ptr(workspace), workspace.numel(), _stream(stream), ctypes.byref(opts))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_index_scores")
    return out


def kpool_balanced_row_split(cu_seqlens, kpool: int, parts: int, row_weight: int = 0) -> list:
    """Bounds [b0=0, b1, ..., b_parts=T] of `parts` contiguous row ranges of near-equal work
    (causal pairs + row_weight per row); cu_seqlens on the host (list, numpy or CPU tensor)."""
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(cu_seqlens if not torch.is_tensor(cu_seqlens) else cu_seqlens.cpu(),
                                         dtype=np.int32))
    out = np.zeros(int(parts) + 1, dtype=np.int32)
    st = load().kpool_balanced_row_split(cu.ctypes.data_as(ctypes.c_void_p), len(cu) - 1, int(kpool),
                                         int(row_weight), int(parts), out.ctypes.data_as(ctypes.c_void_p))
    if st != KPOOL_OK:
        raise KpoolError(st, "kpool_balanced_row_split")
    return [int(x) for x in out]
