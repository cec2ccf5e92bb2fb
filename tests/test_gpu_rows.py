"""GPU parity of kpool_select_rows (explicit query rows against a pooled-key cache: the
decode / short-query case) against the oracle, through the C ABI.

Each row (sequence b, position t) must get exactly what row t of the whole-batch
selection gets for the same query and weights, so the oracle is the same
per-row selection, called with the rows' global indices cu[b] + t and the rows'
own queries.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

CANARY = -7


def _run_rows(wl, inp, kp_gpu=None, row_seq=None, row_pos=None, extra=2):
    """Select through the C ABI into canary-padded buffers; returns (ids, tokens, scores, status)."""
    dev = inp["q"].device
    R, B, Wd = wl.num_rows, wl.budget, wl.width
    if kp_gpu is None:
        kp_gpu = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ids_buf = torch.full((R + extra, B), CANARY, dtype=torch.int32, device=dev)
    tok_buf = torch.full((R + extra, Wd), CANARY, dtype=torch.int32, device=dev)
    sc_buf = torch.full((R + extra, B), float(CANARY), dtype=torch.float32, device=dev)
    ws = K.new_rows_workspace(R, wl.total_tokens, wl.num_seqs, wl.kpool, wl.index_topk, dev)
    K.kpool_select_rows(inp["q"], inp["w"], inp["row_seq"] if row_seq is None else row_seq,
                        inp["row_pos"] if row_pos is None else row_pos, kp_gpu, inp["cu_seqlens"],
                        wl.total_tokens, wl.kpool, wl.index_topk, wl.scale, out_pool_ids=ids_buf[:R],
                        out_token_ids=tok_buf[:R], out_pool_scores=sc_buf[:R], workspace=ws)
    st = K.kpool_last_device_error(ws)
    assert (ids_buf[R:] == CANARY).all() and (tok_buf[R:] == CANARY).all() and (sc_buf[R:] == CANARY).all(), \
        "write past the last row"
    return ids_buf[:R].cpu().numpy(), tok_buf[:R].cpu().numpy(), sc_buf[:R].cpu().numpy(), st


def _oracle_rows(wl, inp):
    cu = inp["cu_seqlens"].cpu().numpy()
    kp = oracle.pool(parity.bits(inp["k"]), wl.dtype, cu, wl.kpool)
    rows = np.array(wl.global_rows(), dtype=np.int64)
    ref = oracle.select(parity.bits(inp["q"]), inp["w"].cpu().numpy(), kp, cu, rows, wl.dtype, wl.kpool,
                        wl.index_topk, wl.scale)
    ref["kp"] = kp
    ref["rows"] = rows
    return ref


def test_rows_float_parity():
    wl = W.DECODE_SMALL
    inp = W.generate_rows(wl, "cuda")
    ids, toks, sc, st = _run_rows(wl, inp)
    assert st == K.KPOOL_OK
    ref = _oracle_rows(wl, inp)
    parity.compare_float({"cu_seqlens": inp["cu_seqlens"]}, wl, ref, ids, sc, toks, q_rows=inp["q"],
                         w_rows=inp["w"])
    # the -1 slots carry -inf scores
    assert np.all(np.isneginf(sc[ids < 0]))


def test_rows_integer_exact():
    wl = W.DECODE_TIE
    inp = W.generate_rows(wl, "cuda")
    ids, toks, sc, st = _run_rows(wl, inp)
    assert st == K.KPOOL_OK
    ref = _oracle_rows(wl, inp)
    parity.assert_exact(ref, ids, toks)
    m = ref["pool_ids"] >= 0
    np.testing.assert_array_equal(sc[m], ref["scores"][m].astype(np.float32))


def test_rows_equal_batch_rows_on_integer_data():
    """Rows picked out of a packed batch give the batch selection's rows, bit for bit."""
    wl = W.TIE_HEAVY
    inp = W.generate(wl, "cuda")
    ids_all, tok_all, _ = K.kpool_select(inp["q"], inp["k"], inp["w"], inp["cu_seqlens"], wl.kpool, wl.index_topk,
                                         wl.scale)
    rows = torch.tensor([0, 3, 4, 2047, 2048, 4095, 4096, 4099, 6000, 8191], dtype=torch.int64)
    cu = inp["cu_seqlens"].cpu()
    b = torch.searchsorted(cu, rows, right=True) - 1
    rwl = W.RowsWorkload("pick", wl.seqlens, tuple((int(x), int(r - cu[x])) for x, r in zip(b, rows)),
                         wl.heads, wl.head_dim, wl.kpool, wl.index_topk, wl.scale, wl.dtype, wl.values, 0)
    rinp = {"k": inp["k"], "cu_seqlens": inp["cu_seqlens"], "q": inp["q"][rows.cuda()].contiguous(),
            "w": inp["w"][rows.cuda()].contiguous(), "row_seq": b.to(torch.int32).cuda(),
            "row_pos": (rows - cu[b]).to(torch.int32).cuda()}
    ids, toks, _, st = _run_rows(rwl, rinp)
    assert st == K.KPOOL_OK
    np.testing.assert_array_equal(ids, ids_all[rows.cuda()].cpu().numpy())
    np.testing.assert_array_equal(toks, tok_all[rows.cuda()].cpu().numpy())


def test_rows_equal_batch_rows_on_float_data():
    """Both score kernels run the same tcgen05 contraction (K = 128 in the same eight K = 16
    steps) and the same fp32 epilogue, so decode rows reproduce the batch selection bit for
    bit on float data too: ids, tokens and scores."""
    wl = W.custom("pickf", (3000, 17, 2100), 32, 128, 4, 2048, 1.0 / np.sqrt(128), "bf16", "normal", 31)
    inp = {k: v.cuda() for k, v in W.generate(wl, "cpu").items()}
    ids_all, tok_all, sc_all = K.kpool_select_ex(inp["q"], inp["k"], inp["w"], inp["cu_seqlens"], wl.kpool,
                                                 wl.index_topk, wl.scale, return_scores=True,
                                                 score_kernel=K.KPOOL_SCORE_TC)
    rows = torch.arange(0, wl.total_tokens, 7)
    cu = inp["cu_seqlens"].cpu()
    b = torch.searchsorted(cu, rows, right=True) - 1
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ids, toks, sc = K.kpool_select_rows(inp["q"][rows.cuda()].contiguous(), inp["w"][rows.cuda()].contiguous(),
                                        b.to(torch.int32).cuda(), (rows - cu[b]).to(torch.int32).cuda(), kp,
                                        inp["cu_seqlens"], wl.total_tokens, wl.kpool, wl.index_topk, wl.scale,
                                        return_scores=True)
    torch.cuda.synchronize()
    r = rows.cuda()
    assert torch.equal(ids, ids_all[r]) and torch.equal(toks, tok_all[r]) and torch.equal(sc, sc_all[r])


def test_rows_invalid_rows_are_empty_and_reported():
    wl = W.DECODE_TIE
    inp = W.generate_rows(wl, "cuda")
    row_seq = inp["row_seq"].clone()
    row_pos = inp["row_pos"].clone()
    row_seq[1] = wl.num_seqs          # no such sequence
    row_pos[3] = wl.seqlens[int(row_seq[3])]  # one past the sequence's end
    ids, toks, sc, st = _run_rows(wl, inp, row_seq=row_seq, row_pos=row_pos)
    assert st == K.KPOOL_ERR_INVALID_ARG
    for r in (1, 3):
        assert (ids[r] == -1).all() and (toks[r] == -1).all() and np.isneginf(sc[r]).all()
    ref = _oracle_rows(wl, inp)
    for r in (0, 2, 4, 5):
        np.testing.assert_array_equal(ids[r], ref["pool_ids"][r])
        np.testing.assert_array_equal(toks[r], ref["token_ids"][r])


def test_rows_malformed_cu_seqlens():
    wl = W.DECODE_TIE
    inp = W.generate_rows(wl, "cuda")
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    bad = dict(inp)
    bad["cu_seqlens"] = torch.tensor([0, 5000, 4096 + 6000 - 1], dtype=torch.int32, device="cuda")
    ids, toks, sc, st = _run_rows(wl, bad, kp_gpu=kp)
    assert st == K.KPOOL_ERR_INVALID_ARG
    assert (ids == -1).all() and (toks == -1).all()


def test_rows_zero_rows_is_a_noop():
    wl = W.DECODE_TIE
    inp = W.generate_rows(wl, "cuda")
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    e = torch.empty((0,), dtype=torch.int32, device="cuda")
    out = K.kpool_select_rows(inp["q"][:0], inp["w"][:0], e, e, kp, inp["cu_seqlens"], wl.total_tokens, wl.kpool,
                              wl.index_topk, wl.scale, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert out[0].shape == (0, wl.budget)


def test_rows_repeated_calls_reuse_workspace():
    """A second call on the same workspace (fewer rows, other positions) is not affected by the first."""
    wl = W.DECODE_SMALL
    inp = W.generate_rows(wl, "cuda")
    ids1, toks1, _, _ = _run_rows(wl, inp)
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ws = K.new_rows_workspace(wl.num_rows, wl.total_tokens, wl.num_seqs, wl.kpool, wl.index_topk)
    for sel in (slice(0, 16), slice(5, 9), slice(0, 16)):
        q, w = inp["q"][sel].contiguous(), inp["w"][sel].contiguous()
        rs, rp = inp["row_seq"][sel].contiguous(), inp["row_pos"][sel].contiguous()
        ids, toks, _ = K.kpool_select_rows(q, w, rs, rp, kp, inp["cu_seqlens"], wl.total_tokens, wl.kpool,
                                           wl.index_topk, wl.scale, workspace=ws)
        assert K.kpool_last_device_error(ws) == K.KPOOL_OK
        np.testing.assert_array_equal(ids.cpu().numpy(), ids1[sel])
        np.testing.assert_array_equal(toks.cpu().numpy(), toks1[sel])


def test_rows_decode_262k_full_size():
    """The decode batch at full size: 16 rows x 65,536 pools, every row checked against the oracle."""
    wl = W.DECODE_262K
    inp = W.generate_rows(wl, "cuda")
    ids, toks, sc, st = _run_rows(wl, inp)
    assert st == K.KPOOL_OK
    ref = _oracle_rows(wl, inp)
    parity.compare_float({"cu_seqlens": inp["cu_seqlens"]}, wl, ref, ids, sc, toks, q_rows=inp["q"],
                         w_rows=inp["w"])


def test_rows_equal_scores_take_the_smallest_pools():
    """All weights zero: every eligible pool scores 0, so the row keeps its budget smallest pool
    indices. The threshold bins of the three rows hold 1,000 and 3,000 tied pools (gathered and
    cut in shared memory) and 8,192 (too many to gather: a search over the whole row)."""
    base = W.DECODE_TIE
    wl = W.RowsWorkload("zero_w", (40000,), ((0, 4000), (0, 11999), (0, 32767)), 32, 128, 4, 2048, 1.0 / 16.0,
                        "bf16", "integer", 21)
    inp = W.generate_rows(wl, "cuda")
    inp["w"].zero_()
    ids, toks, sc, st = _run_rows(wl, inp)
    assert st == K.KPOOL_OK
    ref = _oracle_rows(wl, inp)
    parity.assert_exact(ref, ids, toks)
    for r in range(3):
        np.testing.assert_array_equal(ids[r], np.arange(wl.budget, dtype=np.int32))
    assert base.budget == wl.budget


@pytest.mark.parametrize("max_ctas", [1, 3, 7, 40])
def test_rows_any_score_grid_gives_the_same_result(max_ctas):
    """The score kernel splits the rows' pools into contiguous runs per CTA; any split
    (one CTA for everything, runs crossing row boundaries) gives identical output."""
    wl = W.DECODE_SMALL
    inp = W.generate_rows(wl, "cuda")
    ids_ref, toks_ref, sc_ref, _ = _run_rows(wl, inp)
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ids, toks, sc = K.kpool_select_rows(inp["q"], inp["w"], inp["row_seq"], inp["row_pos"], kp, inp["cu_seqlens"],
                                        wl.total_tokens, wl.kpool, wl.index_topk, wl.scale, return_scores=True,
                                        max_ctas=max_ctas)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_array_equal(toks.cpu().numpy(), toks_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)


def test_rows_graph_replay_equals_eager():
    """The step captured into a CUDA graph (the score, collect and select kernels then
    hang off programmatic edges) and replayed gives the eager result every time."""
    wl = W.DECODE_SMALL
    inp = W.generate_rows(wl, "cuda")
    ids_ref, toks_ref, sc_ref, _ = _run_rows(wl, inp)
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ws = K.new_rows_workspace(wl.num_rows, wl.total_tokens, wl.num_seqs, wl.kpool, wl.index_topk)
    ids = torch.empty((wl.num_rows, wl.budget), dtype=torch.int32, device="cuda")
    toks = torch.empty((wl.num_rows, wl.width), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.num_rows, wl.budget), dtype=torch.float32, device="cuda")
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        with torch.cuda.graph(graph, stream=gs):
            K.kpool_select_rows(inp["q"], inp["w"], inp["row_seq"], inp["row_pos"], kp, inp["cu_seqlens"],
                                wl.total_tokens, wl.kpool, wl.index_topk, wl.scale, out_pool_ids=ids,
                                out_token_ids=toks, out_pool_scores=sc, workspace=ws, stream=gs)
    torch.cuda.current_stream().wait_stream(gs)
    for _ in range(3):
        ids.fill_(CANARY)
        toks.fill_(CANARY)
        graph.replay()
        torch.cuda.synchronize()
        assert K.kpool_last_device_error(ws) == K.KPOOL_OK
        np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
        np.testing.assert_array_equal(toks.cpu().numpy(), toks_ref)
        np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)
