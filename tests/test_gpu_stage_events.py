"""The per-kernel stage events of the _ex entry points: recorded around every kernel of a
call, launched directly or replayed from a captured CUDA graph (inside a capture the
library adds them as event-record nodes), without changing any result."""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _events(n, stream):
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in ev:
        e.record(stream)
    return ev


def _stage_ms(ev):
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(len(ev) - 1)]


def test_batch_stage_events_eager():
    wl = W.TIE_HEAVY
    inp = W.generate(wl, "cuda")
    stream = torch.cuda.current_stream()
    ref_ids, ref_tok, _ = K.kpool_select(inp["q"], inp["k"], inp["w"], inp["cu_seqlens"], wl.kpool, wl.index_topk,
                                         wl.scale)
    ev = _events(5, stream)
    ids, tok, _ = K.kpool_select_ex(inp["q"], inp["k"], inp["w"], inp["cu_seqlens"], wl.kpool, wl.index_topk,
                                    wl.scale, stream=stream, stage_events=ev)
    torch.cuda.synchronize()
    ms = _stage_ms(ev)
    assert all(t >= 0.0 for t in ms) and ms[2] > 0.0  # plan, pool, score+select, expand
    assert abs(sum(ms) - ev[0].elapsed_time(ev[4])) < 1e-2
    assert torch.equal(ids, ref_ids) and torch.equal(tok, ref_tok)


def test_rows_stage_events_in_a_captured_graph():
    wl = W.DECODE_SMALL
    inp = W.generate_rows(wl, "cuda")
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ws = K.new_rows_workspace(wl.num_rows, wl.total_tokens, wl.num_seqs, wl.kpool, wl.index_topk)
    ids = torch.empty((wl.num_rows, wl.budget), dtype=torch.int32, device="cuda")
    tok = torch.empty((wl.num_rows, wl.width), dtype=torch.int32, device="cuda")

    def call(stream, ev=None):
        K.kpool_select_rows(inp["q"], inp["w"], inp["row_seq"], inp["row_pos"], kp, inp["cu_seqlens"],
                            wl.total_tokens, wl.kpool, wl.index_topk, wl.scale, out_pool_ids=ids, out_token_ids=tok,
                            workspace=ws, stream=stream, stage_events=ev)

    call(torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref_ids, ref_tok = ids.clone(), tok.clone()
    ids.fill_(-7)
    tok.fill_(-7)
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    ev = _events(4, torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        with torch.cuda.graph(graph, stream=gs):
            call(gs, ev)
    torch.cuda.current_stream().wait_stream(gs)
    for _ in range(3):
        ids.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        ms = _stage_ms(ev)
        assert all(t >= 0.0 for t in ms) and ms[1] > 0.0  # plan, score, collect + select
        assert K.kpool_last_device_error(ws) == K.KPOOL_OK
        np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy())
        np.testing.assert_array_equal(tok.cpu().numpy(), ref_tok.cpu().numpy())
