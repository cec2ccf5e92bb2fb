"""The parity rules themselves: the comparison helpers accept the oracle's own answer
and reject each kind of wrong answer a kernel could give (CPU only; the "GPU" output is
the oracle's, with one planted mistake at a time)."""
import numpy as np
import pytest

from sparse_attention_kpool_gb300 import workloads as W
from tests import parity


@pytest.fixture(scope="module")
def case():
    wl = W.TINY
    inp = W.generate(wl, "cpu")
    rows = np.arange(wl.total_tokens, dtype=np.int64)
    ref = parity.oracle_rows(inp, wl, rows)
    return wl, inp, ref


def _copy(ref):
    return ref["pool_ids"].copy(), ref["scores"].astype(np.float32), ref["token_ids"].copy()


def _full_row(ref, B):
    """A row whose budget is full and whose cutoff is clear of the next pool."""
    for i in range(len(ref["rows"]) - 1, -1, -1):
        if (ref["pool_ids"][i] >= 0).sum() == B:
            return i
    raise AssertionError("no full row")


def test_oracle_answer_passes_float_rule(case):
    wl, inp, ref = case
    ids, sc, tok = _copy(ref)
    stats = parity.compare_float(inp, wl, ref, ids, sc, tok)
    assert stats["rows"] == wl.total_tokens and stats["near_tie_rows"] == 0
    parity.assert_exact(ref, ids, tok)


def _rejects(case, mutate):
    wl, inp, ref = case
    ids, sc, tok = _copy(ref)
    mutate(wl, ref, ids, sc, tok)
    with pytest.raises(AssertionError):
        parity.compare_float(inp, wl, ref, ids, sc, tok)


def test_rejects_a_pool_far_below_the_cutoff(case):
    from oracle import oracle
    wl, inp, ref = case
    i = _full_row(ref, wl.budget)
    t = int(ref["rows"][i])
    e = (t + 1) // wl.kpool
    qr, wr = parity.bits(inp["q"][t]), inp["w"][t].numpy()
    unchosen = [p for p in range(e) if p not in set(ref["pool_ids"][i].tolist())]
    scores = {p: oracle.score(qr, wr, ref["kp"][p], wl.dtype, wl.scale) for p in unchosen}
    worst = min(unchosen, key=lambda p: scores[p])
    cut = float(ref["scores"][i, wl.budget - 1])
    assert scores[worst] < cut - parity._tol(ref["scores"][i], cut)  # a real error, not a near tie

    def m(wl, ref, ids, sc, tok):
        ids[i, wl.budget - 1] = worst
        sc[i, wl.budget - 1] = scores[worst]
        tok[i, (wl.budget - 1) * wl.kpool:wl.budget * wl.kpool] = worst * wl.kpool + np.arange(wl.kpool)
    _rejects(case, m)


def test_rejects_a_wrong_score(case):
    def m(wl, ref, ids, sc, tok):
        i = _full_row(ref, wl.budget)
        sc[i, 0] = sc[i, 0] * 1.01 + 1e-3
    _rejects(case, m)


def test_rejects_a_repeated_pool(case):
    def m(wl, ref, ids, sc, tok):
        i = _full_row(ref, wl.budget)
        ids[i, 1] = ids[i, 0]
        tok[i, wl.kpool:2 * wl.kpool] = tok[i, 0:wl.kpool]
    _rejects(case, m)


def test_rejects_an_ineligible_pool(case):
    def m(wl, ref, ids, sc, tok):
        i = _full_row(ref, wl.budget)
        t = int(ref["rows"][i])
        e = (t + 1) // wl.kpool
        ids[i, wl.budget - 1] = e  # the row's own, not yet complete (or future) pool
        tok[i, (wl.budget - 1) * wl.kpool:wl.budget * wl.kpool] = e * wl.kpool + np.arange(wl.kpool)
    _rejects(case, m)


def test_rejects_a_wrong_expanded_token(case):
    def m(wl, ref, ids, sc, tok):
        i = _full_row(ref, wl.budget)
        tok[i, 1] += 1
    _rejects(case, m)


def test_rejects_a_wrong_tail(case):
    def m(wl, ref, ids, sc, tok):
        i = next(i for i in range(len(ref["rows"])) if (int(ref["rows"][i]) + 1) % wl.kpool != 0)
        tok[i, wl.budget * wl.kpool] = -1 if tok[i, wl.budget * wl.kpool] >= 0 else 0
    _rejects(case, m)


def test_rejects_a_missing_pool(case):
    def m(wl, ref, ids, sc, tok):
        i = _full_row(ref, wl.budget)
        ids[i, wl.budget - 1] = -1
        tok[i, (wl.budget - 1) * wl.kpool:wl.budget * wl.kpool] = -1
    _rejects(case, m)


def test_rejects_a_reversed_order(case):
    def m(wl, ref, ids, sc, tok):
        i = _full_row(ref, wl.budget)
        ids[i, [0, wl.budget - 1]] = ids[i, [wl.budget - 1, 0]]
        sc[i, [0, wl.budget - 1]] = sc[i, [wl.budget - 1, 0]]
        for j in (0, wl.budget - 1):
            tok[i, j * wl.kpool:(j + 1) * wl.kpool] = ids[i, j] * wl.kpool + np.arange(wl.kpool)
    _rejects(case, m)


def test_exact_rule_rejects_any_change(case):
    wl, inp, ref = case
    ids, sc, tok = _copy(ref)
    i = _full_row(ref, wl.budget)
    ids[i, [0, 1]] = ids[i, [1, 0]]
    with pytest.raises(AssertionError):
        parity.assert_exact(ref, ids, tok)


# ---------------------------------------------------- a packed batch of two sequences
#
# The rule works in sequence-local indices: the eligibility bound comes from the row's
# own sequence in cu_seqlens, the oracle's pools are offset by that sequence's first
# pool, and the expanded tokens count from the sequence's first token. Mistakes planted
# in the second sequence (nonzero offsets) must be caught as well.

@pytest.fixture(scope="module")
def packed_case():
    wl = W.custom("packed2", (41, 58), heads=4, head_dim=32, kpool=4, index_topk=16, scale=0.17,
                  dtype="f32", values="normal", seed=9)
    inp = W.generate(wl, "cpu")
    rows = np.arange(wl.total_tokens, dtype=np.int64)
    ref = parity.oracle_rows(inp, wl, rows)
    return wl, inp, ref


def _second_seq_full_row(wl, inp, ref):
    cu = inp["cu_seqlens"].numpy()
    for i in range(len(ref["rows"]) - 1, -1, -1):
        if int(ref["rows"][i]) >= cu[1] and (ref["pool_ids"][i] >= 0).sum() == wl.budget:
            return i, int(ref["rows"][i]) - int(cu[1])
    raise AssertionError("no full row in the second sequence")


def test_packed_oracle_answer_passes(packed_case):
    wl, inp, ref = packed_case
    ids, sc, tok = _copy(ref)
    assert parity.compare_float(inp, wl, ref, ids, sc, tok)["near_tie_rows"] == 0


def test_packed_rejects_batch_global_pool_ids(packed_case):
    wl, inp, ref = packed_case
    first_pool = int(inp["cu_seqlens"][1]) // wl.kpool  # pools of the first sequence
    ids, sc, tok = _copy(ref)
    i, _ = _second_seq_full_row(wl, inp, ref)
    ids[i] = ids[i] + first_pool
    tok[i, :wl.budget * wl.kpool] = (ids[i][:, None] * wl.kpool + np.arange(wl.kpool)).ravel()
    with pytest.raises(AssertionError):
        parity.compare_float(inp, wl, ref, ids, sc, tok)


def test_packed_rejects_batch_global_token_ids(packed_case):
    wl, inp, ref = packed_case
    ids, sc, tok = _copy(ref)
    i, _ = _second_seq_full_row(wl, inp, ref)
    first_token = int(inp["cu_seqlens"][1])
    tok[i, :wl.budget * wl.kpool] += first_token
    with pytest.raises(AssertionError):
        parity.compare_float(inp, wl, ref, ids, sc, tok)


def test_packed_rejects_a_pool_just_past_the_rows_bound(packed_case):
    wl, inp, ref = packed_case
    ids, sc, tok = _copy(ref)
    i, t = _second_seq_full_row(wl, inp, ref)
    e = (t + 1) // wl.kpool  # sequence-local eligible pools of that row
    ids[i, wl.budget - 1] = e
    tok[i, (wl.budget - 1) * wl.kpool:wl.budget * wl.kpool] = e * wl.kpool + np.arange(wl.kpool)
    with pytest.raises(AssertionError):
        parity.compare_float(inp, wl, ref, ids, sc, tok)


def test_packed_rejects_scores_of_the_wrong_sequence(packed_case):
    """A kernel that scored the second sequence's row against the first sequence's pools."""
    from oracle import oracle
    wl, inp, ref = packed_case
    ids, sc, tok = _copy(ref)
    i, t = _second_seq_full_row(wl, inp, ref)
    row = int(ref["rows"][i])
    qr, wr = parity.bits(inp["q"][row]), inp["w"][row].numpy()
    sc[i, :wl.budget] = [oracle.score(qr, wr, ref["kp"][int(p)], wl.dtype, wl.scale) for p in ids[i]]
    with pytest.raises(AssertionError):
        parity.compare_float(inp, wl, ref, ids, sc, tok)
