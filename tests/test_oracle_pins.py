"""Pins for the CPU oracle: checks against what the pages and the mathematics fix,
never against the oracle itself.

* hand-worked golden cases (tests/golden/*.json, each citing its page/section);
* brute force on the Tiny workload by an independent numpy/itertools restatement
  that picks the top set by enumerating every subset;
* special cases that reduce to textbook routines (H=1, w=1, scale=1 -> relu(q.K^T)
  ranked by numpy; kpool=1 -> the per-token indexer);
* closed forms (mean of integer keys), invariants and metamorphic relations
  (head permutation, packed vs alone, row sub-ranges).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_attention_kpool_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element storage for the oracle: bf16 as uint16 bit patterns, fp32 as float32."""
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.to(torch.float32).numpy()


def values(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def run_oracle(inp: dict, wl: W.Workload, lib=None) -> dict:
    return oracle.select_all(bits(inp["q"]), bits(inp["k"]), inp["w"].numpy(),
                             inp["cu_seqlens"].numpy(), wl.dtype, wl.kpool, wl.index_topk, wl.scale,
                             lib=lib)


def expand_ranges(ranges, n_rows):
    out = [None] * n_rows
    for lo, hi, ids in ranges:
        for t in range(lo, hi + 1):
            out[t] = ids
    assert all(o is not None for o in out)
    return np.array(out, dtype=np.int32)


# ---------------------------------------------------------------- golden cases

def _const_pool_inputs(pool_values, seqlen, kpool, d, channel0_only=True):
    keys = np.zeros((seqlen, d), dtype=np.float32)
    for p, v in enumerate(pool_values):
        keys[p * kpool:(p + 1) * kpool, 0] = v
    return keys


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_golden_tie_straddles_cutoff(dtype, lib=None):
    g = json.load(open(os.path.join(GOLDEN, "tie_straddles_cutoff.json")))
    L, kpool, d, H = g["seqlens"][0], g["kpool"], g["head_dim"], g["heads"]
    keys = _const_pool_inputs(g["pool_values"], L, kpool, d)
    q = np.tile(np.array(g["query"], dtype=np.float32), (L, H, 1))
    w = np.full((L, H), g["weight"], dtype=np.float32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = oracle.select_all(bits(torch.from_numpy(q).to(tdt)), bits(torch.from_numpy(keys).to(tdt)), w,
                            np.array([0, L], dtype=np.int32), dtype, kpool, g["index_topk"], g["scale"],
                            lib=lib)
    want = expand_ranges(g["expected_pool_ids_by_row_range"], L)
    np.testing.assert_array_equal(out["pool_ids"], want)
    for t, row in g["expected_token_rows"].items():
        np.testing.assert_array_equal(out["token_ids"][int(t)], np.array(row, dtype=np.int32))


def test_golden_signs_and_scale(lib=None):
    g = json.load(open(os.path.join(GOLDEN, "signs_and_scale.json")))
    L, kpool, d, H = g["seqlens"][0], g["kpool"], g["head_dim"], g["heads"]
    keys = _const_pool_inputs(g["pool_values"], L, kpool, d)
    q = np.tile(np.array(g["queries_per_head"], dtype=np.float32)[None], (L, 1, 1))
    for case in g["cases"]:
        w = np.tile(np.array(case["weights"], dtype=np.float32), (L, 1))
        out = oracle.select_all(q, keys, w, np.array([0, L], dtype=np.int32), "f32", kpool,
                                g["index_topk"], g["scale"], lib=lib)
        np.testing.assert_array_equal(out["pool_ids"], expand_ranges(case["expected_pool_ids_by_row_range"], L))
        # the last row sees every pool: its selected scores are the hand-derived ones
        last = out["pool_ids"][-1]
        np.testing.assert_array_equal(out["scores"][-1], np.array(case["scores"], dtype=np.float64)[last])


def test_golden_varlen_tail_kpool3(lib=None):
    g = json.load(open(os.path.join(GOLDEN, "varlen_tail_kpool3.json")))
    kpool = g["kpool"]
    keys = np.array(g["keys"], dtype=np.float32)[:, None]
    T = len(keys)
    cu = np.cumsum([0] + g["seqlens"]).astype(np.int32)
    q = np.ones((T, 1, 1), dtype=np.float32)
    w = np.ones((T, 1), dtype=np.float32)
    kp = oracle.pool(keys, "f32", cu, kpool, lib=lib)
    np.testing.assert_array_equal(kp[:, 0], np.array(g["expected_pooled_keys"], dtype=np.float32))
    out = oracle.select_all(q, keys, w, cu, "f32", kpool, g["index_topk"], g["scale"], lib=lib)
    np.testing.assert_array_equal(out["pool_ids"], np.array(g["expected_pool_ids"], dtype=np.int32))
    np.testing.assert_array_equal(out["token_ids"], np.array(g["expected_token_ids"], dtype=np.int32))


def test_golden_per_token_kpool1(lib=None):
    g = json.load(open(os.path.join(GOLDEN, "per_token_kpool1.json")))
    keys = np.array(g["keys"], dtype=np.float32)[:, None]
    T = len(keys)
    out = oracle.select_all(np.ones((T, 1, 1), np.float32), keys, np.ones((T, 1), np.float32),
                            np.array([0, T], dtype=np.int32), "f32", g["kpool"], g["index_topk"], g["scale"],
                            lib=lib)
    np.testing.assert_array_equal(out["pool_ids"], np.array(g["expected_pool_ids"], dtype=np.int32))
    np.testing.assert_array_equal(out["token_ids"], np.array(g["expected_token_ids"], dtype=np.int32))


def test_golden_bf16_pool_rounding(lib=None):
    g = json.load(open(os.path.join(GOLDEN, "bf16_pool_rounding.json")))
    kpool = g["kpool"]
    keys = np.array([c["keys"] for c in g["cases"]], dtype=np.float32).reshape(-1, 1)
    kb = torch.from_numpy(keys).to(torch.bfloat16)
    assert torch.equal(kb.float(), torch.from_numpy(keys)), "fixture keys must be exact bf16 values"
    kp = oracle.pool(bits(kb), "bf16", np.array([0, len(keys)], dtype=np.int32), kpool, lib=lib)
    np.testing.assert_array_equal(kp[:, 0], np.array([c["pooled"] for c in g["cases"]], dtype=np.float32))


# ------------------------------------------------------- independent brute force

def brute_pool(k: np.ndarray, cu, kpool: int, dtype: str) -> np.ndarray:
    """Mean of kpool keys: fp32 adds in key order, one fp32 division, then torch's own
    float->bf16 conversion (round to nearest even) for bf16 inputs."""
    rows = []
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        for p in range((e - s) // kpool):
            acc = np.zeros(k.shape[1], dtype=np.float32)
            for j in range(kpool):
                acc = (acc + k[s + p * kpool + j].astype(np.float32)).astype(np.float32)
            m = (acc / np.float32(kpool)).astype(np.float32)
            if dtype == "bf16":
                m = torch.from_numpy(m).to(torch.bfloat16).to(torch.float32).numpy()
            rows.append(m)
    return np.array(rows, dtype=np.float32).reshape(-1, k.shape[1])


def brute_scores(qv: np.ndarray, wv: np.ndarray, kp: np.ndarray, scale: float) -> np.ndarray:
    """[rows, pools] = sum_h w * relu(scale * q_h . kp) via einsum in fp64. The scale is
    an fp32 argument of the operation, so its fp32 value is the one used."""
    dots = np.einsum("thc,pc->thp", qv.astype(np.float64), kp.astype(np.float64))
    s = np.float64(np.float32(scale))
    return np.einsum("th,thp->tp", wv.astype(np.float64), np.maximum(s * dots, 0.0))


def best_subset(scores: np.ndarray, m: int):
    """The size-m subset whose keys (score, -index), listed best first, are
    lexicographically largest -- found by enumerating every subset."""
    best, best_key = None, None
    for sub in itertools.combinations(range(len(scores)), m):
        key = sorted(((scores[p], -p) for p in sub), reverse=True)
        if best_key is None or key > best_key:
            best, best_key = [-kk[1] for kk in key], key
    return best or []


def test_brute_force_tiny(lib=None):
    wl = W.TINY
    inp = W.generate(wl, "cpu")
    out = run_oracle(inp, wl, lib)
    q, k, w = values(inp["q"]), values(inp["k"]), inp["w"].numpy()
    cu = inp["cu_seqlens"].numpy()
    kp = brute_pool(k.astype(np.float32), cu, wl.kpool, wl.dtype)
    np.testing.assert_array_equal(out["kp"], kp)
    S = brute_scores(q, w, kp, wl.scale)
    B = wl.budget
    for t in range(wl.total_tokens):
        e = (t + 1) // wl.kpool
        m = min(B, e)
        chosen = best_subset(S[t, :e], m)
        want = np.array(chosen + [-1] * (B - m), dtype=np.int32)
        np.testing.assert_array_equal(out["pool_ids"][t], want, err_msg=f"row {t}")
        np.testing.assert_allclose(out["scores"][t, :m], S[t, chosen], rtol=1e-12, atol=1e-12)
        toks = [p * wl.kpool + r if p >= 0 else -1 for p in want for r in range(wl.kpool)]
        tail = (t + 1) % wl.kpool
        toks += [e * wl.kpool + r if r < tail else -1 for r in range(wl.kpool)]
        np.testing.assert_array_equal(out["token_ids"][t], np.array(toks, dtype=np.int32))


def rank_by_numpy(scores: np.ndarray, m: int) -> np.ndarray:
    """Indices of the m best entries under (score desc, index asc), via np.lexsort."""
    order = np.lexsort((np.arange(len(scores)), -scores))
    return order[:m]


def test_h1_unit_weight_reduces_to_relu_qk(lib=None):
    """H=1, w=1, scale=1: the score is relu(q . kpool), ranked by numpy's matmul + lexsort."""
    wl = W.custom("h1", (300,), heads=1, head_dim=16, kpool=4, index_topk=32, scale=1.0, dtype="bf16",
                  values="integer", seed=21)
    inp = W.generate(wl, "cpu")
    inp["w"] = torch.ones_like(inp["w"])
    out = run_oracle(inp, wl, lib)
    kp = brute_pool(values(inp["k"]).astype(np.float32), inp["cu_seqlens"].numpy(), wl.kpool, "bf16")
    rel = np.maximum(values(inp["q"])[:, 0, :] @ kp.astype(np.float64).T, 0.0)
    B = wl.budget
    for t in range(wl.total_tokens):
        e = (t + 1) // wl.kpool
        m = min(B, e)
        want = np.concatenate([rank_by_numpy(rel[t, :e], m), -np.ones(B - m, dtype=np.int64)])
        np.testing.assert_array_equal(out["pool_ids"][t], want.astype(np.int32), err_msg=f"row {t}")


def test_kpool1_is_per_token_indexer(lib=None):
    """kpool=1: pools are single keys, every key up to the row is eligible, no tail."""
    wl = W.custom("k1", (97, 40), heads=3, head_dim=8, kpool=1, index_topk=12, scale=0.5, dtype="f32",
                  values="normal", seed=22)
    inp = W.generate(wl, "cpu")
    out = run_oracle(inp, wl, lib)
    cu = inp["cu_seqlens"].numpy()
    q, k, w = values(inp["q"]), values(inp["k"]), inp["w"].numpy()
    for b in range(wl.num_seqs):
        s, e_ = int(cu[b]), int(cu[b + 1])
        S = brute_scores(q[s:e_], w[s:e_], k[s:e_], wl.scale)
        for t in range(e_ - s):
            m = min(wl.budget, t + 1)
            want = np.concatenate([rank_by_numpy(S[t, :t + 1], m), -np.ones(wl.budget - m, dtype=np.int64)])
            np.testing.assert_array_equal(out["pool_ids"][s + t], want.astype(np.int32))
            assert (out["token_ids"][s + t, wl.budget:] == -1).all()


# ------------------------------------------------- closed forms and invariants

@pytest.mark.parametrize("kpool", [3, 4, 5])
def test_pool_mean_closed_form_on_integers(kpool, lib=None):
    """Integer keys: the pooled value is fp32(exact sum) / kpool correctly rounded; with
    kpool a power of two the result is the exact rational mean."""
    wl = W.custom("pc", (61, 0, 29), heads=1, head_dim=24, kpool=kpool, index_topk=kpool, scale=1.0,
                  dtype="f32", values="integer", seed=23)
    inp = W.generate(wl, "cpu")
    k = values(inp["k"])
    cu = inp["cu_seqlens"].numpy()
    kp = oracle.pool(bits(inp["k"]), "f32", cu, kpool, lib=lib)
    r = 0
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        for p in range((e - s) // kpool):
            for c in range(k.shape[1]):
                exact = Fraction(int(sum(k[s + p * kpool + j, c] for j in range(kpool))), kpool)
                got = Fraction(float(kp[r, c]))
                if kpool & (kpool - 1) == 0:
                    assert got == exact
                else:
                    # correctly rounded to fp32: within half an ulp of the exact mean
                    half_ulp = Fraction(float(np.spacing(np.abs(np.float32(kp[r, c]))))) / 2
                    assert abs(got - exact) <= half_ulp
            r += 1
    assert r == kp.shape[0]


def check_invariants(out: dict, cu: np.ndarray, kpool: int, index_topk: int):
    B = index_topk // kpool
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        L = e - s
        for t in range(L):
            ids = out["pool_ids"][s + t]
            el = (t + 1) // kpool
            m = min(B, el)
            assert (ids[:m] >= 0).all() and (ids[m:] == -1).all(), f"padding at row {s + t}"
            assert (ids[:m] < el).all(), "pool beyond the row"
            assert len(set(ids[:m].tolist())) == m, "duplicate pool"
            sc = out["scores"][s + t, :m]
            assert (np.diff(sc) <= 0).all(), "not in rank order"
            for j in range(m - 1):
                if sc[j] == sc[j + 1]:
                    assert ids[j] < ids[j + 1], "tie not broken toward the smaller index"
            tok = out["token_ids"][s + t]
            valid = tok[tok >= 0]
            assert (valid <= t).all() and (valid < L).all()
            assert len(set(valid.tolist())) == len(valid)
            tail = tok[B * kpool:]
            assert (tail >= 0).sum() == (t + 1) % kpool


@pytest.mark.parametrize("seed", [31, 32])
def test_invariants_ragged_packed(seed, lib=None):
    wl = W.custom("inv", (1, 3, 0, 37, 130, 64, 5), heads=4, head_dim=16, kpool=4, index_topk=24, scale=0.3,
                  dtype="bf16", values="normal", seed=seed)
    inp = W.generate(wl, "cpu")
    out = run_oracle(inp, wl, lib)
    check_invariants(out, inp["cu_seqlens"].numpy(), wl.kpool, wl.index_topk)


def test_budget_covers_all_eligible_pools():
    wl = W.custom("all", (50,), heads=2, head_dim=8, kpool=4, index_topk=64, scale=1.0, dtype="f32",
                  values="normal", seed=33)
    inp = W.generate(wl, "cpu")
    out = run_oracle(inp, wl)
    for t in range(50):
        el = (t + 1) // 4
        assert sorted(out["pool_ids"][t, :el].tolist()) == list(range(el))
        assert (out["pool_ids"][t, el:] == -1).all()


def test_short_rows_and_empty_sequences(lib=None):
    wl = W.custom("short", (0, 2, 3, 0, 1), heads=2, head_dim=8, kpool=4, index_topk=8, scale=1.0,
                  dtype="f32", values="normal", seed=34)
    inp = W.generate(wl, "cpu")
    out = run_oracle(inp, wl, lib)
    assert (out["pool_ids"] == -1).all()
    cu = inp["cu_seqlens"].numpy()
    for b in range(len(cu) - 1):
        for t in range(int(cu[b + 1] - cu[b])):
            tok = out["token_ids"][cu[b] + t]
            assert tok[:8].tolist() == [-1] * 8
            assert tok[8:].tolist() == [r if r <= t else -1 for r in range(4)]


def test_head_permutation_invariance():
    wl = W.custom("perm", (200,), heads=8, head_dim=16, kpool=4, index_topk=20, scale=1.0 / 16, dtype="bf16",
                  values="integer", seed=35)
    inp = W.generate(wl, "cpu")
    base = run_oracle(inp, wl)
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(5))
    inp2 = dict(inp, q=inp["q"][:, perm].contiguous(), w=inp["w"][:, perm].contiguous())
    out = run_oracle(inp2, wl)
    np.testing.assert_array_equal(out["pool_ids"], base["pool_ids"])
    np.testing.assert_array_equal(out["scores"], base["scores"])


def test_packed_equals_alone(lib=None):
    wl = W.custom("pack", (45, 90, 17), heads=4, head_dim=16, kpool=4, index_topk=16, scale=0.25,
                  dtype="bf16", values="integer", seed=36)
    inp = W.generate(wl, "cpu")
    packed = run_oracle(inp, wl, lib)
    cu = inp["cu_seqlens"].numpy()
    for b in range(3):
        s, e = int(cu[b]), int(cu[b + 1])
        alone = oracle.select_all(bits(inp["q"][s:e]), bits(inp["k"][s:e]), inp["w"][s:e].numpy(),
                                  np.array([0, e - s], dtype=np.int32), wl.dtype, wl.kpool, wl.index_topk,
                                  wl.scale, lib=lib)
        np.testing.assert_array_equal(packed["pool_ids"][s:e], alone["pool_ids"])
        np.testing.assert_array_equal(packed["token_ids"][s:e], alone["token_ids"])


def test_row_subranges_concatenate():
    """Rows are independent: scoring row ranges separately and concatenating equals the whole
    (the pages' query-row shard test, on one process)."""
    wl = W.custom("split", (37, 24, 5), heads=4, head_dim=16, kpool=4, index_topk=12, scale=0.5,
                  dtype="bf16", values="normal", seed=37)
    inp = W.generate(wl, "cpu")
    whole = run_oracle(inp, wl)
    kp = oracle.pool(bits(inp["k"]), "bf16", inp["cu_seqlens"].numpy(), wl.kpool)
    T = wl.total_tokens
    for G in (2, 3, 8):
        per = -(-T // G)
        parts = []
        for r in range(G):
            rows = np.arange(r * per, min(T, (r + 1) * per), dtype=np.int64)
            part = oracle.select(bits(inp["q"][rows]), inp["w"][rows].numpy(), kp, inp["cu_seqlens"].numpy(),
                                 rows, "bf16", wl.kpool, wl.index_topk, wl.scale)
            parts.append(part["pool_ids"])
        np.testing.assert_array_equal(np.concatenate(parts), whole["pool_ids"])


def test_tie_heavy_recipe_has_cutoff_ties():
    """The tie-heavy recipe really produces exact ties that straddle the budget cutoff."""
    wl = W.custom("ties", (512,), heads=32, head_dim=128, kpool=4, index_topk=64, scale=1.0 / 16,
                  dtype="bf16", values="integer", seed=2, dup_every=8)
    inp = W.generate(wl, "cpu")
    out = run_oracle(inp, wl)
    check_invariants(out, inp["cu_seqlens"].numpy(), wl.kpool, wl.index_topk)
    kp = out["kp"]
    q, w = values(inp["q"]), inp["w"].numpy()
    S = brute_scores(q, w, kp, wl.scale)
    straddling = 0
    for t in range(wl.total_tokens):
        el = (t + 1) // wl.kpool
        if el <= wl.budget:
            continue
        ids = out["pool_ids"][t]
        cut = S[t, ids[-1]]
        unchosen = np.setdiff1d(np.arange(el), ids)
        if (S[t, unchosen] == cut).any():
            straddling += 1
            # every unchosen pool tied with the cutoff has a larger index than the chosen ones at that score
            tied_in = ids[S[t, ids] == cut]
            assert unchosen[S[t, unchosen] == cut].min() > tied_in.max()
    assert straddling > 0


# ---- gated pooling (a stated reading of the pages' compress gate / position embedding)
#
# kp[p,c] = sum_j softmax_j(gate[t_j,c]) * (k[t_j,c] + ape[j,c]); the pins below fix it
# by hand-worked values, by its reduction to the mean, and by a one-hot gate that must
# pick exactly one position per channel.

def _bits_bf16(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_pool_hand_example(dtype, lib=None):
    # one pool of two tokens, two channels: channel 0 weights (3/4, 1/4), channel 1 (1/4, 3/4)
    k = torch.tensor([[4.0, 8.0], [8.0, 16.0]])
    gate = np.array([[math.log(3.0), 0.0], [0.0, math.log(3.0)]], dtype=np.float32)
    ape = np.array([[1.0, 0.0], [0.0, 2.0]], dtype=np.float32)
    kk = _bits_bf16(k) if dtype == "bf16" else k.numpy()
    out = oracle.pool_gated(kk, gate, ape, dtype, np.array([0, 2], dtype=np.int32), 2, lib=lib)
    # 3/4 (4 + 1) + 1/4 (8 + 0) = 5.75 and 1/4 (8 + 0) + 3/4 (16 + 2) = 15.5
    np.testing.assert_allclose(out, [[5.75, 15.5]], rtol=1e-6)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gated_pool_zero_gate_zero_ape_is_the_mean(dtype, lib=None):
    g = torch.Generator().manual_seed(31)
    cu = np.array([0, 37, 37, 100], dtype=np.int32)
    k = torch.randint(-2, 3, (100, 8), generator=g).to(torch.float32)
    kk = _bits_bf16(k) if dtype == "bf16" else k.numpy()
    for kpool in (1, 3, 4):
        gated = oracle.pool_gated(kk, np.zeros((100, 8), np.float32), np.zeros((kpool, 8), np.float32), dtype, cu,
                                  kpool, lib=lib)
        np.testing.assert_array_equal(gated, oracle.pool(kk, dtype, cu, kpool, lib=lib))


def test_gated_pool_one_hot_gate_picks_a_position(lib=None):
    """A gate that is 0 at one position and -1e4 elsewhere makes the softmax one-hot: the
    pooled channel is that token's key plus that position's embedding (channel c picks
    position c mod kpool, so a position/channel mix-up shows)."""
    kpool, d, T = 4, 8, 24
    g = torch.Generator().manual_seed(5)
    k = torch.randn((T, d), generator=g)
    ape = torch.randn((kpool, d), generator=g).numpy()
    gate = np.full((T, d), -1e4, dtype=np.float32)
    for t in range(T):
        for c in range(d):
            if t % kpool == c % kpool:
                gate[t, c] = 0.0
    out = oracle.pool_gated(k.numpy(), gate, ape, "f32", np.array([0, T], dtype=np.int32), kpool, lib=lib)
    kn = k.numpy()
    for p in range(T // kpool):
        for c in range(d):
            j = c % kpool
            assert out[p, c] == np.float32(np.float64(kn[p * kpool + j, c]) + np.float64(ape[j, c]))


def test_gated_pool_shift_invariance(lib=None):
    """Adding a constant to a pool's gate scores (per channel) leaves the softmax unchanged."""
    kpool, d, T = 4, 16, 64
    g = torch.Generator().manual_seed(8)
    k = _bits_bf16(torch.randn((T, d), generator=g))
    gate = (torch.randn((T, d), generator=g) * 2).numpy()
    ape = (torch.randn((kpool, d), generator=g) * 0.1).numpy()
    cu = np.array([0, T], dtype=np.int32)
    a = oracle.pool_gated(k, gate, ape, "bf16", cu, kpool, lib=lib)
    b = oracle.pool_gated(k, gate + np.float32(3.0), ape, "bf16", cu, kpool, lib=lib)
    np.testing.assert_array_equal(a, b)


def test_tie_heavy_full_budget_has_cutoff_ties():
    """At its full size and budget (2 x 4096 tokens, budget 512) the tie-heavy workload has
    rows where an exact tie straddles the cutoff, so its bit-exact GPU comparison exercises
    the smaller-index tiebreak at budget 512. Checked on a few of those rows by brute force."""
    from tests import parity
    wl = W.TIE_HEAVY
    inp = W.generate(wl, "cpu")
    cu = inp["cu_seqlens"].numpy()
    kp = oracle.pool(bits(inp["k"]), wl.dtype, cu, wl.kpool)
    q, w = values(inp["q"]), inp["w"].numpy()
    wide = oracle.select(bits(inp["q"]), w, kp, cu, np.arange(wl.total_tokens), wl.dtype, wl.kpool,
                         wl.index_topk + wl.kpool, wl.scale)
    rows = parity.cutoff_tie_rows(wide, wl.budget)
    assert len(rows) > 0
    for i in rows[:: max(1, len(rows) // 5)][:5]:
        t = int(i)
        b = int(np.searchsorted(cu, t, side="right") - 1)
        e = (t - int(cu[b]) + 1) // wl.kpool
        pool0 = int(oracle.pool_offsets(cu, wl.kpool)[b])
        s = brute_scores(q[t:t + 1], w[t:t + 1], kp[pool0:pool0 + e], wl.scale)[0]
        order = np.lexsort((np.arange(e), -s))  # score descending, then pool ascending
        np.testing.assert_array_equal(order[:wl.budget + 1], wide["pool_ids"][i])
        assert s[order[wl.budget - 1]] == s[order[wl.budget]]
