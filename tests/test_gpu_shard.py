"""Query-row sharding on one GPU: every simulated rank's row range through the C ABI.

The pages test their query split in a single process against the unsharded call,
bitwise ("NVIDIA/Megatron-LM pull request #8299", section "Test plan"). Here each
rank's kpool_select_ex with a row range is run in turn on one GPU, and the
concatenation of the shards' pool ids and token ids must equal the unsharded
call's bit for bit -- for 2, 3 and 8 ranks, for the pair-balanced split and the
pages' even row split, with ragged and empty shards, on a packed (THD) batch, on
both score kernels, and on float as well as integer data (rows are independent,
so a row's result cannot depend on which shard computes it). Expanding the
concatenated pool ids with kpool_expand must give the same token ids again, as
the gathered path does after its all-gather.
"""
import numpy as np
import pytest
import torch

from sparse_attention_kpool_gb300 import build as kbuild
from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import shard
from sparse_attention_kpool_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    kbuild.build()
    K.load()


def _even_rows(T, G):
    step = -(-T // G)  # the pages' split: rank r takes rows [r * ceil(T/G), ...)
    return [min(T, r * step) for r in range(G)] + [T]


@pytest.mark.parametrize("values", ["integer", "normal"])
@pytest.mark.parametrize("kernel", [K.KPOOL_SCORE_TC, K.KPOOL_SCORE_SIMT])
def test_shards_concatenate_to_the_unsharded_call(values, kernel):
    wl = W.custom("shard", (3001, 17, 0, 9000, 7, 2500), 32, 128, 4, 2048,
                  1.0 / 16 if values == "integer" else 1.0 / np.sqrt(128), "bf16", values, 81,
                  dup_every=8 if values == "integer" else 0)
    dev = {k: v.cuda() for k, v in W.generate(wl, "cpu").items()}
    T = wl.total_tokens
    ws = K.new_workspace(T, wl.num_seqs, 32, 128, K.KPOOL_BF16, wl.kpool, wl.index_topk)
    ids, toks, _ = K.kpool_select_ex(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk,
                                     wl.scale, workspace=ws, score_kernel=kernel)
    torch.cuda.synchronize()
    ids, toks = ids.cpu(), toks.cpu()
    cu = dev["cu_seqlens"].cpu()
    splits = []
    for G in (2, 3, 8):
        splits.append(shard.row_bounds(cu, wl.kpool, G))
        splits.append(_even_rows(T, G))
    splits.append([0, 0, 5, 5, 3018, T, T])  # empty first, ragged and empty shards, a cut at a sequence end
    for bounds in splits:
        parts_ids, parts_toks = [], []
        for lo, hi in zip(bounds, bounds[1:]):
            if hi == lo:
                continue
            i, t, _ = K.kpool_select_ex(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk,
                                        wl.scale, workspace=ws, score_kernel=kernel, row_range=(lo, hi))
            assert i.shape == (hi - lo, wl.budget) and t.shape == (hi - lo, wl.width)
            parts_ids.append(i)
            parts_toks.append(t)
        torch.cuda.synchronize()
        assert K.kpool_last_device_error(ws) == K.KPOOL_OK
        got_ids = torch.cat(parts_ids).cpu()
        np.testing.assert_array_equal(got_ids.numpy(), ids.numpy(), err_msg=f"pool ids, bounds {bounds}")
        np.testing.assert_array_equal(torch.cat(parts_toks).cpu().numpy(), toks.numpy(),
                                      err_msg=f"token ids, bounds {bounds}")
        re_toks = K.kpool_expand(got_ids.cuda(), dev["cu_seqlens"], wl.kpool, wl.index_topk)
        np.testing.assert_array_equal(re_toks.cpu().numpy(), toks.numpy())


def test_a_shard_writes_only_its_own_rows():
    """Output buffers sized for the shard, with canaries on both sides: nothing outside."""
    wl = W.custom("shardc", (700, 333), 32, 128, 4, 256, 1.0 / 16, "bf16", "integer", 82)
    dev = {k: v.cuda() for k, v in W.generate(wl, "cpu").items()}
    lo, hi = 501, 909  # straddles the sequence boundary at 700, not a multiple of the 8-row item
    R, B, Wd, pad = hi - lo, wl.budget, wl.width, 4096
    ids_buf = torch.full((R * B + 2 * pad,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    tok_buf = torch.full((R * Wd + 2 * pad,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    ids = ids_buf[pad:pad + R * B].view(R, B)
    toks = tok_buf[pad:pad + R * Wd].view(R, Wd)
    K.kpool_select_ex(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk, wl.scale,
                      out_pool_ids=ids, out_token_ids=toks, row_range=(lo, hi))
    full_ids, full_toks, _ = K.kpool_select_ex(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool,
                                               wl.index_topk, wl.scale)
    torch.cuda.synchronize()
    for buf in (ids_buf, tok_buf):
        assert bool((buf[:pad] == 0x5A5A5A5A).all()) and bool((buf[-pad:] == 0x5A5A5A5A).all())
    assert torch.equal(ids, full_ids[lo:hi]) and torch.equal(toks, full_toks[lo:hi])


def test_sharded_path_rejects_index_scores():
    wl = W.custom("shards", (64,), 32, 128, 4, 64, 1.0 / 16, "bf16", "integer", 83)
    dev = {k: v.cuda() for k, v in W.generate(wl, "cpu").items()}
    with pytest.raises(K.KpoolError) as e:
        K.kpool_select_ex(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk, wl.scale,
                          return_scores=True, row_range=(0, 32))
    assert e.value.status == K.KPOOL_ERR_INVALID_ARG
