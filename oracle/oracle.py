"""ctypes wrapper around the CPU oracle (kpool_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this module; the product path never does. It shares no
code with the CUDA library. Inputs are numpy arrays; bf16 tensors travel as
their raw uint16 bit patterns.

The method it restates (mean pooling of kpool keys, the head-weighted relu
score, top-budget selection with ties to the smaller pool index, expansion,
tail append and mask) is documented step by step at the top of
kpool_oracle.c, with the page and section each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kpool_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkpool_oracle.so")

DTYPES = {"bf16": 0, "f32": 1}

_lib = None
_lock = threading.Lock()


def compile_source(src: str, out_path: str) -> str:
    """Compile one oracle C source with the oracle's flags (used for the oracle itself and
    for the planted-mistake copies the tests build)."""
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
         "-Wall", "-Wextra", "-o", tmp, src, "-lm"],
        check=True,
    )
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction) and return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def open_library(path: str):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    lib.kpool_oracle_pool_offsets.argtypes = [P, i32, i32, P]
    lib.kpool_oracle_pool_offsets.restype = i32
    lib.kpool_oracle_pool.argtypes = [P, i32, P, i32, i32, i32, P]
    lib.kpool_oracle_pool.restype = i32
    lib.kpool_oracle_pool_gated.argtypes = [P, i32, P, P, P, i32, i32, i32, P]
    lib.kpool_oracle_pool_gated.restype = i32
    lib.kpool_oracle_score.argtypes = [P, i32, P, P, i32, i32, ctypes.c_float]
    lib.kpool_oracle_score.restype = ctypes.c_double
    lib.kpool_oracle_select.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32,
                                        ctypes.c_float, P, i64, P, P, P, P]
    lib.kpool_oracle_select.restype = i32
    lib.kpool_oracle_threads.argtypes = []
    lib.kpool_oracle_threads.restype = i32
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _elem(a: np.ndarray, dtype: str) -> np.ndarray:
    want = np.uint16 if dtype == "bf16" else np.float32
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"{dtype} data must arrive as {np.dtype(want).name}, got {a.dtype}")
    return a


def threads(lib=None) -> int:
    return int(_load(lib).kpool_oracle_threads())


def pool_offsets(cu_seqlens: np.ndarray, kpool: int, lib=None) -> np.ndarray:
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    out = np.zeros(len(cu), dtype=np.int64)
    rc = _load(lib).kpool_oracle_pool_offsets(_ptr(cu), len(cu) - 1, kpool, _ptr(out))
    if rc != 0:
        raise ValueError("invalid cu_seqlens / kpool")
    return out


def pool(k: np.ndarray, dtype: str, cu_seqlens: np.ndarray, kpool: int, lib=None) -> np.ndarray:
    """Mean-pooled keys [P, d] as float32 values (already rounded to the input dtype)."""
    k = _elem(k, dtype)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    d = k.shape[-1]
    P = int(pool_offsets(cu, kpool, lib)[-1])
    out = np.zeros((P, d), dtype=np.float32)
    rc = _load(lib).kpool_oracle_pool(_ptr(k), DTYPES[dtype], _ptr(cu), len(cu) - 1, d, kpool, _ptr(out))
    if rc != 0:
        raise ValueError("invalid pooling arguments")
    return out


def pool_gated(k: np.ndarray, gate: np.ndarray, ape: np.ndarray, dtype: str, cu_seqlens: np.ndarray, kpool: int,
               lib=None) -> np.ndarray:
    """Gated pooled keys [P, d] (float32 values rounded to the input dtype): per pool and channel a
    softmax over the pool's positions of gate [T, d] weights k + ape (ape [kpool, d])."""
    k = _elem(k, dtype)
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    ape = np.ascontiguousarray(ape, dtype=np.float32)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    d = k.shape[-1]
    if gate.shape != (k.shape[0], d) or ape.shape != (kpool, d):
        raise ValueError("gate must be [T, d] and ape [kpool, d]")
    P = int(pool_offsets(cu, kpool, lib)[-1])
    out = np.zeros((P, d), dtype=np.float32)
    rc = _load(lib).kpool_oracle_pool_gated(_ptr(k), DTYPES[dtype], _ptr(gate), _ptr(ape), _ptr(cu), len(cu) - 1, d,
                                            kpool, _ptr(out))
    if rc != 0:
        raise ValueError("invalid pooling arguments")
    return out


def score(q_row: np.ndarray, w_row: np.ndarray, kp_row: np.ndarray, dtype: str, scale: float,
          lib=None) -> float:
    """fp64 score of one (query row, pool): q_row [H, d], w_row [H], kp_row [d]."""
    q_row = _elem(q_row, dtype)
    w_row = np.ascontiguousarray(w_row, dtype=np.float32)
    kp_row = np.ascontiguousarray(kp_row, dtype=np.float32)
    H, d = q_row.shape
    return float(_load(lib).kpool_oracle_score(_ptr(q_row), DTYPES[dtype], _ptr(w_row), _ptr(kp_row),
                                            H, d, scale))


def select(q_rows: np.ndarray, w_rows: np.ndarray, kp: np.ndarray, cu_seqlens: np.ndarray,
           rows: np.ndarray, dtype: str, kpool: int, index_topk: int, scale: float, lib=None) -> dict:
    """Selection for the listed global rows.

    q_rows [n, H, d] (bf16 bits or f32) and w_rows [n, H] f32 hold the listed rows'
    queries and weights; kp [P, d] comes from pool(). Returns pool_ids [n, B],
    token_ids [n, index_topk + kpool], scores [n, B] (fp64, NaN on -1 slots) and
    eligible [n].
    """
    q_rows = _elem(q_rows, dtype)
    w_rows = np.ascontiguousarray(w_rows, dtype=np.float32)
    kp = np.ascontiguousarray(kp, dtype=np.float32)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = len(rows)
    H, d = q_rows.shape[-2], q_rows.shape[-1]
    if kpool < 1 or index_topk % kpool:
        raise ValueError("index_topk must be a multiple of kpool >= 1")
    B = index_topk // kpool
    W = index_topk + kpool
    pool_ids = np.empty((n, B), dtype=np.int32)
    token_ids = np.empty((n, W), dtype=np.int32)
    scores = np.empty((n, B), dtype=np.float64)
    eligible = np.empty((n,), dtype=np.int64)
    rc = _load(lib).kpool_oracle_select(
        _ptr(q_rows), _ptr(w_rows), _ptr(kp), _ptr(cu), len(cu) - 1, H, d, DTYPES[dtype], kpool,
        index_topk, scale, _ptr(rows), n, _ptr(pool_ids), _ptr(token_ids), _ptr(scores),
        _ptr(eligible))
    if rc != 0:
        raise ValueError("invalid selection arguments")
    return {"pool_ids": pool_ids, "token_ids": token_ids, "scores": scores, "eligible": eligible}


def select_all(q: np.ndarray, k: np.ndarray, w: np.ndarray, cu_seqlens: np.ndarray, dtype: str,
               kpool: int, index_topk: int, scale: float, lib=None) -> dict:
    """Every row of a packed batch: q [T, H, d], k [T, d], w [T, H]."""
    kp = pool(k, dtype, cu_seqlens, kpool, lib)
    T = q.shape[0]
    out = select(q, w, kp, cu_seqlens, np.arange(T, dtype=np.int64), dtype, kpool, index_topk, scale,
                 lib)
    out["kp"] = kp
    return out
