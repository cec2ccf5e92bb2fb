"""Comparison helpers for GPU-vs-oracle parity.

Bit-exact comparison for integer-valued inputs; for float inputs the rule is:
  * every GPU pool score is within TOL_REL * max(|s_ref|, 1e-3 * rowmax|s_ref|)
    of the oracle's fp64 score of the same (row, pool);
  * the number of chosen pools and the tail match exactly;
  * the chosen pools are distinct and causally eligible, and the expanded token
    slots follow the GPU's own pool ids exactly;
  * the chosen set equals the oracle's, except that every pool in the symmetric
    difference scores (per the oracle) within that tolerance of the row's
    cutoff score -- near-ties may go either way;
  * the GPU order is non-increasing in oracle score up to the tolerance.
TOL_REL is the stated score tolerance: 1e-3 relative error at fp32 accumulation.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle

TOL_REL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.to(torch.float32).numpy()


def oracle_rows(inp: dict, wl, rows: np.ndarray, kp: np.ndarray | None = None) -> dict:
    """Oracle selection for the listed global rows (inputs may live on the GPU)."""
    rows = np.asarray(rows, dtype=np.int64)
    ridx = torch.as_tensor(rows, device=inp["q"].device)
    cu = inp["cu_seqlens"].cpu().numpy()
    if kp is None:
        kp = oracle.pool(bits(inp["k"]), wl.dtype, cu, wl.kpool)
    out = oracle.select(bits(inp["q"][ridx]), inp["w"][ridx].cpu().numpy(), kp, cu, rows, wl.dtype, wl.kpool,
                        wl.index_topk, wl.scale)
    out["kp"] = kp
    out["rows"] = rows
    return out


def _tol(s_ref_row: np.ndarray, s: float) -> float:
    rowmax = float(np.nanmax(np.abs(s_ref_row))) if np.isfinite(s_ref_row).any() else 0.0
    return TOL_REL * max(abs(s), 1e-3 * rowmax, 1e-30)


def compare_float(inp: dict, wl, ref: dict, gpu_ids: np.ndarray, gpu_scores: np.ndarray | None,
                  gpu_tokens: np.ndarray, q_rows=None, w_rows=None) -> dict:
    """Apply the tolerance rule to the rows in ref["rows"]; returns counters. Raises AssertionError.

    The query and weights of ref row i are inp["q"][row], inp["w"][row] (a packed batch), or
    q_rows[i], w_rows[i] when those are given (explicit query rows)."""
    cu = inp["cu_seqlens"].cpu().numpy()
    kp = ref["kp"]
    B = wl.budget
    near_tie_rows = 0
    max_rel_err = 0.0    # largest |s_gpu - s_ref| / max(|s_ref|, 1e-3 rowmax) seen
    scores_compared = 0
    q_cpu_cache = {}
    for i, row in enumerate(ref["rows"]):
        rid, gid = ref["pool_ids"][i], gpu_ids[i]
        m = int((rid >= 0).sum())
        assert int((gid >= 0).sum()) == m, f"row {row}: {int((gid >= 0).sum())} pools chosen, oracle {m}"
        assert (gid[m:] == -1).all()
        # tail slots are pure index arithmetic: exact
        np.testing.assert_array_equal(gpu_tokens[i, B * wl.kpool:], ref["token_ids"][i, B * wl.kpool:],
                                      err_msg=f"row {row}: tail")
        # the expanded slots follow the GPU's own pool ids exactly
        kpl = np.arange(wl.kpool, dtype=np.int64)
        expect = np.where(gid[:, None] >= 0, gid[:, None].astype(np.int64) * wl.kpool + kpl, -1).ravel()
        np.testing.assert_array_equal(gpu_tokens[i, :B * wl.kpool], expect, err_msg=f"row {row}: expanded slots")
        if m == 0:
            continue
        # chosen pools are distinct and causally eligible for this row
        b_row = int(np.searchsorted(cu, row, side="right") - 1)
        e_row = (int(row) - int(cu[b_row]) + 1) // wl.kpool
        assert len(set(gid[:m].tolist())) == m, f"row {row}: repeated pool ids"
        assert int(gid[:m].max()) < e_row, f"row {row}: pool {int(gid[:m].max())} is not eligible (e = {e_row})"
        if np.array_equal(rid, gid):
            same = True
        else:
            same = False
        b = int(np.searchsorted(cu, row, side="right") - 1)
        pool0 = int(oracle.pool_offsets(cu, wl.kpool)[b])
        if q_rows is not None:
            qr, wr = bits(q_rows[i]), w_rows[i].cpu().numpy()
        else:
            if row not in q_cpu_cache:
                q_cpu_cache[row] = (bits(inp["q"][row]), inp["w"][row].cpu().numpy())
            qr, wr = q_cpu_cache[row]

        def s_ref(p):
            return oracle.score(qr, wr, kp[pool0 + p], wl.dtype, wl.scale)

        ref_scores = ref["scores"][i, :m]
        cut = float(ref_scores[m - 1])
        tol = _tol(ref_scores, cut)
        if gpu_scores is not None:
            for j in range(m):
                sr = float(ref_scores[j]) if same else s_ref(int(gid[j]))
                err = abs(float(gpu_scores[i, j]) - sr)
                assert err <= _tol(ref_scores, sr), \
                    f"row {row} slot {j}: gpu score {gpu_scores[i, j]} vs oracle {sr}"
                max_rel_err = max(max_rel_err, err / (_tol(ref_scores, sr) / TOL_REL))
                scores_compared += 1
        if same:
            continue
        g_set, r_set = set(gid[:m].tolist()), set(rid[:m].tolist())
        for p in g_set ^ r_set:
            sp = s_ref(int(p))
            assert abs(sp - cut) <= tol, f"row {row}: pool {p} (oracle score {sp}) differs beyond the cutoff band"
        g_sc = [s_ref(int(p)) for p in gid[:m]]
        for j in range(m - 1):
            assert g_sc[j] >= g_sc[j + 1] - _tol(ref_scores, g_sc[j]), f"row {row}: order at slot {j}"
        near_tie_rows += 1
    return {"rows": len(ref["rows"]), "near_tie_rows": near_tie_rows, "max_rel_err": max_rel_err,
            "scores_compared": scores_compared}


def oracle_full_scores(inp: dict, wl, rows: np.ndarray, ld: int, kp: np.ndarray | None = None) -> np.ndarray:
    """The oracle's fp64 score of every pool of the listed global rows as an [n, ld] matrix,
    -inf where the pool is not eligible: the oracle's selection with a budget as large as
    the batch's pool count keeps (and scores) every eligible pool of a row."""
    rows = np.asarray(rows, dtype=np.int64)
    cu = inp["cu_seqlens"].cpu().numpy()
    if kp is None:
        kp = oracle.pool(bits(inp["k"]), wl.dtype, cu, wl.kpool)
    every = max(1, wl.total_tokens // wl.kpool)
    ridx = torch.as_tensor(rows, device=inp["q"].device)
    sel = oracle.select(bits(inp["q"][ridx]), inp["w"][ridx].cpu().numpy(), kp, cu, rows, wl.dtype, wl.kpool,
                        wl.kpool * every, wl.scale)
    full = np.full((len(rows), ld), -np.inf)
    for i in range(len(rows)):
        ids = sel["pool_ids"][i]
        m = ids >= 0
        assert int(m.sum()) == int(sel["eligible"][i])
        keep = ids[m] < ld
        full[i, ids[m][keep]] = sel["scores"][i, m][keep]
    return full


def compare_full_scores(gpu: np.ndarray, ref: np.ndarray, exact: bool, what: str = "") -> float:
    """Index scores against the oracle's: -inf in exactly the same places, and every finite
    score equal (exact) or within TOL_REL * max(|s_ref|, 1e-3 * rowmax |s_ref|). Returns the
    largest relative error seen."""
    assert gpu.shape == ref.shape
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(np.isfinite(gpu), fin, err_msg=f"{what}: eligible pattern")
    assert (gpu[~fin] == -np.inf).all(), f"{what}: non-eligible pools must be -inf"
    if exact:
        np.testing.assert_array_equal(gpu[fin].astype(np.float64), ref[fin], err_msg=f"{what}: scores")
        return 0.0
    rowmax = np.max(np.where(fin, np.abs(ref), 0.0), axis=1, keepdims=True)
    base = np.maximum(np.maximum(np.abs(ref), 1e-3 * rowmax), 1e-30)[fin]
    err = np.abs(gpu.astype(np.float64)[fin] - ref[fin]) / base
    worst = float(err.max()) if err.size else 0.0
    assert worst <= TOL_REL, f"{what}: relative score error {worst:.3e} > {TOL_REL}"
    return worst


def cutoff_tie_rows(ref_wide: dict, budget: int) -> np.ndarray:
    """Rows (indices into ref_wide) where an exact tie straddles the budget cutoff: the
    budget-th and (budget+1)-th ranked scores are equal, so the tiebreak alone decides
    which pool is kept. ref_wide is an oracle selection with at least budget + 1 slots."""
    sc = ref_wide["scores"]
    assert sc.shape[1] > budget
    both = (ref_wide["pool_ids"][:, budget - 1] >= 0) & (ref_wide["pool_ids"][:, budget] >= 0)
    return np.nonzero(both & (sc[:, budget - 1] == sc[:, budget]))[0]


def assert_exact(ref: dict, gpu_ids: np.ndarray, gpu_tokens: np.ndarray):
    for i, row in enumerate(ref["rows"]):
        np.testing.assert_array_equal(gpu_ids[i], ref["pool_ids"][i], err_msg=f"pool ids, row {row}")
        np.testing.assert_array_equal(gpu_tokens[i], ref["token_ids"][i], err_msg=f"token ids, row {row}")
