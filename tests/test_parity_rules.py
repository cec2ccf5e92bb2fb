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
