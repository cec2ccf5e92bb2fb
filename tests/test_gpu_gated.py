"""GPU parity of the gated pooling (kpool_pool_keys_gated) and of the selection from given
pooled keys (kpool_select_pooled) against the oracle, through the C ABI.

Gated pooling runs in fp32 on the GPU and in fp64 in the oracle, so a pooled key may land
one unit in the last place of the key dtype apart; the selection is then checked with the
stated score tolerance. With a zero gate and embedding the gated keys must equal the mean
pooling bit for bit, and selecting from the library's own mean-pooled keys must equal the
whole-batch call bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


def _gate_ape(wl, T, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    gate = (torch.randn((T, wl.head_dim), generator=g) * 2.0).cuda()
    ape = (torch.randn((wl.kpool, wl.head_dim), generator=g) * 0.25).cuda()
    return gate, ape


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), np.float32(2.0 ** -126))))
    return np.exp2(e - 7)


@pytest.mark.parametrize("name", ["varlen", "tie_heavy"])
def test_gated_pooled_keys_match_oracle(name):
    wl = W.BY_NAME[name]
    inp = W.generate(wl, "cuda")
    gate, ape = _gate_ape(wl, wl.total_tokens, 17)
    kp = K.kpool_pool_keys_gated(inp["k"], gate, ape, inp["cu_seqlens"], wl.kpool)
    cu = inp["cu_seqlens"].cpu().numpy()
    ref = oracle.pool_gated(parity.bits(inp["k"]), gate.cpu().numpy(), ape.cpu().numpy(), wl.dtype, cu, wl.kpool)
    P = ref.shape[0]
    got = kp[:P].float().cpu().numpy()
    # bound: fp32 evaluation of a kpool-term weighted sum (a few units of 2^-24 of the
    # largest term) plus one bf16 rounding step on each side
    k = inp["k"].float().cpu().numpy()
    a = ape.cpu().numpy()
    terms = np.zeros_like(ref)
    for b in range(wl.num_seqs):
        n = (int(cu[b + 1]) - int(cu[b])) // wl.kpool
        p0 = int(oracle.pool_offsets(cu, wl.kpool)[b])
        for j in range(wl.kpool):
            x = np.abs(k[int(cu[b]) + j: int(cu[b]) + n * wl.kpool: wl.kpool] + a[j])
            terms[p0:p0 + n] = np.maximum(terms[p0:p0 + n], x)
    bound = _bf16_ulp(ref) + 1e-6 * terms
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"worst excess {np.max(err - bound)} at {np.unravel_index(np.argmax(err - bound), err.shape)}"
    assert (err == 0).mean() > 0.99


def test_gated_zero_gate_is_mean_pooling_bit_for_bit():
    wl = W.VARLEN
    inp = W.generate(wl, "cuda")
    T, d = inp["k"].shape
    kp_mean = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    kp_gated = K.kpool_pool_keys_gated(inp["k"], torch.zeros((T, d), device="cuda"),
                                       torch.zeros((wl.kpool, d), device="cuda"), inp["cu_seqlens"], wl.kpool)
    assert torch.equal(kp_mean.view(torch.int16), kp_gated.view(torch.int16))


@pytest.mark.parametrize("kernel", [K.KPOOL_SCORE_TC, K.KPOOL_SCORE_SIMT])
def test_select_pooled_equals_whole_call(kernel):
    wl = W.TIE_HEAVY
    inp = W.generate(wl, "cuda")
    ids_a, tok_a, sc_a = K.kpool_select_ex(inp["q"], inp["k"], inp["w"], inp["cu_seqlens"], wl.kpool,
                                           wl.index_topk, wl.scale, return_scores=True, score_kernel=kernel)
    kp = K.kpool_pool_keys(inp["k"], inp["cu_seqlens"], wl.kpool)
    ids_b, tok_b, sc_b = K.kpool_select_pooled(inp["q"], kp, inp["w"], inp["cu_seqlens"], wl.kpool, wl.index_topk,
                                               wl.scale, return_scores=True, score_kernel=kernel)
    assert torch.equal(ids_a, ids_b) and torch.equal(tok_a, tok_b) and torch.equal(sc_a, sc_b)


def test_gated_selection_matches_oracle():
    wl = W.VARLEN
    inp = W.generate(wl, "cuda")
    gate, ape = _gate_ape(wl, wl.total_tokens, 23)
    kp = K.kpool_pool_keys_gated(inp["k"], gate, ape, inp["cu_seqlens"], wl.kpool)
    ids, toks, sc = K.kpool_select_pooled(inp["q"], kp, inp["w"], inp["cu_seqlens"], wl.kpool, wl.index_topk,
                                          wl.scale, return_scores=True)
    # the pooled keys themselves are checked against the oracle above; here the oracle
    # selects from the very keys the GPU used, so only the selection is compared
    P = int(oracle.pool_offsets(inp["cu_seqlens"].cpu().numpy(), wl.kpool)[-1])
    kp_used = kp[:P].float().cpu().numpy()
    rows = W.sample_rows(wl, 400).numpy()
    ref = parity.oracle_rows(inp, wl, rows, kp=kp_used)
    r = torch.as_tensor(rows, device="cuda")
    parity.compare_float(inp, wl, ref, ids[r].cpu().numpy(), sc[r].cpu().numpy(), toks[r].cpu().numpy())
