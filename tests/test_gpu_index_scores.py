"""Full index scores (kpool_index_scores) through the C ABI, against the oracle.

The pages' op can return its index scores, which it computes in row chunks of at
most 2 GiB ("NVIDIA/Megatron-LM pull request #8299", section "Change"). Checked
here: every element of the compared rows against the oracle's fp64 scores (bit for
bit on integer-valued inputs, the stated relative tolerance on float inputs), -inf
in exactly the non-eligible places, chunks that concatenate to the whole call bit
for bit, and agreement with the selection: the scores the selection returns are the
full scores at the chosen pools, bit for bit, and the chosen pools are the top
budget of each full row under "higher score, then smaller pool index"
("spark_model/layers/glm5next_dsa/tp.rs", module docs).
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_attention_kpool_gb300 import build as kbuild
from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

TC, SIMT = K.KPOOL_SCORE_TC, K.KPOOL_SCORE_SIMT
MAX_OBSERVED_REL_ERR = 1e-5  # fp32 accumulation of exact bf16 products: errors stay near 1e-6


@pytest.fixture(scope="module", autouse=True)
def library():
    kbuild.build()
    K.load()
    oracle.build()


def to_dev(inp):
    return {k: v.cuda() for k, v in inp.items()}


def scores(dev, wl, **kw):
    out = K.kpool_index_scores(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.scale, **kw)
    torch.cuda.synchronize()
    return out


def eligible_mask(cu: torch.Tensor, kpool: int, rows: torch.Tensor, ld: int) -> torch.Tensor:
    """[n, ld] bool: pool p is eligible for global row r (p < floor((t+1)/kpool))."""
    cu = cu.long()
    seq = torch.searchsorted(cu[1:], rows, right=True)
    e = (rows - cu[seq] + 1) // kpool
    return torch.arange(ld, device=rows.device)[None, :] < e[:, None]


def _wl(values, seed, seqlens=(3001, 17, 0, 2100, 7), dtype="bf16", heads=32, dim=128):
    scale = 1.0 / 16 if values == "integer" else 1.0 / np.sqrt(dim)
    return W.custom("isc", seqlens, heads, dim, 4, 256, scale, dtype, values, seed)


@pytest.mark.parametrize("values", ["integer", "normal"])
@pytest.mark.parametrize("kernel", [TC, SIMT])
def test_rows_match_the_oracle(values, kernel):
    wl = _wl(values, 90 + kernel)
    inp = W.generate(wl, "cpu")
    dev = to_dev(inp)
    ld = wl.total_tokens // wl.kpool
    full = scores(dev, wl, ld=ld, score_kernel=kernel).cpu().numpy()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(0, 12), np.arange(3001, 3030), rng.integers(0, wl.total_tokens, 160),
                                     np.arange(wl.total_tokens - 9, wl.total_tokens)]))
    ref = parity.oracle_full_scores(dev, wl, rows, ld)
    err = parity.compare_full_scores(full[rows], ref, exact=values == "integer", what=f"{values}/{kernel}")
    print(f"\n{values} kernel {kernel}: {len(rows)} rows x {ld} pools, max relative error {err:.2e}")
    assert err <= MAX_OBSERVED_REL_ERR


@pytest.mark.parametrize("wl", [W.TINY, _wl("normal", 93, seqlens=(700, 333), heads=16, dim=64),
                                _wl("normal", 94, seqlens=(515,), dtype="f32")],
                         ids=["tiny_f32", "h16_d64", "f32_h32"])
def test_simt_shapes_match_the_oracle(wl):
    dev = to_dev(W.generate(wl, "cpu"))
    ld = wl.total_tokens // wl.kpool + 3  # wider than any row: the extra columns are -inf
    full = scores(dev, wl, ld=ld).cpu().numpy()
    rows = np.arange(wl.total_tokens)
    ref = parity.oracle_full_scores(dev, wl, rows, ld)
    parity.compare_full_scores(full, ref, exact=False, what=wl.name)


@pytest.mark.parametrize("kpool", [1, 3, 8])
def test_other_kpool_exact(kpool):
    """Pools of 1, 3 and 8 keys (ragged tails, a sequence shorter than one pool): both
    kernel families against the oracle, bit for bit on integer-valued inputs."""
    wl = W.custom("isc_k", (777, 5, 2, 1300), 32, 128, kpool, 8 * kpool, 1.0 / 16, "bf16", "integer", 100 + kpool)
    dev = to_dev(W.generate(wl, "cpu"))
    ld = max(int(L) // kpool for L in wl.seqlens)
    rows = np.arange(wl.total_tokens)
    ref = parity.oracle_full_scores(dev, wl, rows, ld)
    for kernel in (TC, SIMT):
        full = scores(dev, wl, ld=ld, score_kernel=kernel).cpu().numpy()
        parity.compare_full_scores(full, ref, exact=True, what=f"kpool {kpool}, kernel {kernel}")


def test_negative_scale():
    wl = W.custom("isc_neg", (1500, 260), 32, 128, 4, 256, -1.0 / 16, "bf16", "integer", 95)
    dev = to_dev(W.generate(wl, "cpu"))
    ld = wl.total_tokens // wl.kpool
    for kernel in (TC, SIMT):
        full = scores(dev, wl, ld=ld, score_kernel=kernel).cpu().numpy()
        rows = np.arange(0, wl.total_tokens, 7)
        parity.compare_full_scores(full[rows], parity.oracle_full_scores(dev, wl, rows, ld), exact=True,
                                   what=f"negative scale, kernel {kernel}")


@pytest.mark.parametrize("kernel", [TC, SIMT])
def test_selection_ranks_the_full_scores(kernel):
    """The selection's scores are the full scores at the chosen pools (bit for bit), and the
    chosen pools are each row's top budget under (higher score, smaller pool)."""
    wl = W.custom("isc_sel", (2500, 1200, 64), 32, 128, 4, 512, 1.0 / np.sqrt(128), "bf16", "normal", 96)
    dev = to_dev(W.generate(wl, "cpu"))
    T, B = wl.total_tokens, wl.budget
    ld = T // wl.kpool
    ids, _, sel = K.kpool_select_ex(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk,
                                    wl.scale, return_scores=True, score_kernel=kernel)
    full = scores(dev, wl, ld=ld, score_kernel=kernel)
    ids = ids.long()
    chosen = ids >= 0
    got = torch.gather(full, 1, ids.clamp(min=0))
    assert torch.equal(torch.where(chosen, got, sel), sel), "selected scores differ from the full scores"
    # stable descending sort keeps equal scores in pool order: the selection order exactly
    order = torch.sort(full, dim=1, descending=True, stable=True).indices[:, :B]
    e = eligible_mask(dev["cu_seqlens"], wl.kpool, torch.arange(T, device="cuda"), ld).sum(1)
    want = torch.where(torch.arange(B, device="cuda")[None, :] < e[:, None], order, torch.full_like(order, -1))
    assert torch.equal(want, ids), "the selection is not the top budget of the full scores"


def test_chunks_concatenate_to_the_whole_call():
    wl = _wl("normal", 97)
    dev = to_dev(W.generate(wl, "cpu"))
    T = wl.total_tokens
    ld = T // wl.kpool
    whole = scores(dev, wl, ld=ld)
    ws = K.new_workspace(T, wl.num_seqs, 32, 128, K.KPOOL_BF16, wl.kpool, 0)
    for bounds in ([0, 1000, 3001, 3018, 5118, T], [0, 0, 5, 5, 2999, 4000, T, T], [0, 8, 16, T]):
        parts = []
        for lo, hi in zip(bounds, bounds[1:]):
            if hi > lo:
                parts.append(K.kpool_index_scores(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool,
                                                  wl.scale, ld=ld, row_range=(lo, hi), workspace=ws))
        torch.cuda.synchronize()
        assert K.kpool_last_device_error(ws) == K.KPOOL_OK
        assert torch.equal(torch.cat(parts), whole), f"bounds {bounds}"


@pytest.mark.parametrize("max_ctas", [1, 7, 152])
def test_any_grid_gives_the_same_scores(max_ctas):
    """The persistent kernel's CTAs take work items from a counter: one CTA working
    through every item, or a few, must write the same matrix as the full grid."""
    wl = _wl("normal", 101, seqlens=(1900, 3, 700))
    dev = to_dev(W.generate(wl, "cpu"))
    ld = wl.total_tokens // wl.kpool
    for kernel in (TC, SIMT):
        ref = scores(dev, wl, ld=ld, score_kernel=kernel)
        got = scores(dev, wl, ld=ld, score_kernel=kernel, max_ctas=max_ctas)
        assert torch.equal(got, ref), f"kernel {kernel}, max_ctas {max_ctas}"


def test_chunk_writes_only_its_rows_and_columns():
    """A chunk written into the middle of a larger buffer: the canaries on both sides survive."""
    wl = _wl("integer", 98, seqlens=(900, 500))
    dev = to_dev(W.generate(wl, "cpu"))
    lo, hi, ld, pad = 333, 1111, 300, 1000
    R = hi - lo
    buf = torch.full((R * ld + 2 * pad,), 7.25, dtype=torch.float32, device="cuda")
    out = buf[pad:pad + R * ld]
    K.kpool_index_scores(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.scale, ld=ld, out=out,
                         row_range=(lo, hi))
    whole = scores(dev, wl, ld=ld)
    assert bool((buf[:pad] == 7.25).all()) and bool((buf[-pad:] == 7.25).all())
    assert torch.equal(out.view(R, ld), whole[lo:hi])


def test_narrow_ld_is_reported_and_keeps_the_first_columns():
    wl = _wl("normal", 99, seqlens=(1200,))
    dev = to_dev(W.generate(wl, "cpu"))
    for kernel in (TC, SIMT):
        wide = scores(dev, wl, ld=300, score_kernel=kernel)
        ws = K.new_workspace(wl.total_tokens, 1, 32, 128, K.KPOOL_BF16, wl.kpool, 0)
        narrow = K.kpool_index_scores(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.scale, ld=100,
                                      workspace=ws, score_kernel=kernel)
        torch.cuda.synchronize()
        assert K.kpool_last_device_error(ws) == K.KPOOL_ERR_INVALID_ARG
        assert torch.equal(narrow, wide[:, :100]), f"kernel {kernel}"


def test_pooled_keys_variant_is_identical():
    wl = _wl("normal", 100)
    dev = to_dev(W.generate(wl, "cpu"))
    ld = wl.total_tokens // wl.kpool
    kp = K.kpool_pool_keys(dev["k"], dev["cu_seqlens"], wl.kpool)
    a = scores(dev, wl, ld=ld)
    b = K.kpool_index_scores(dev["q"], kp, dev["w"], dev["cu_seqlens"], wl.kpool, wl.scale, ld=ld, pooled=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_long_128k_last_chunk_full_size():
    """long_128k in the launch configuration the benchmark times: 2 GiB chunks of
    16,384 rows x 32,768 pools. The deepest chunk: sampled rows against the oracle,
    and on every row of it the -inf pattern and non-negative scores (w >= 0)."""
    wl = W.LONG_128K
    dev = W.generate(wl, "cuda")
    T = wl.total_tokens
    ld = T // wl.kpool
    chunk = (2 << 30) // (4 * ld)
    lo, hi = T - chunk, T
    out = K.kpool_index_scores(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.scale, ld=ld,
                               row_range=(lo, hi))
    torch.cuda.synchronize()
    rows = torch.arange(lo, hi, device="cuda")
    fin = torch.isfinite(out)
    assert torch.equal(fin, eligible_mask(dev["cu_seqlens"], wl.kpool, rows, ld)), "eligible pattern"
    assert bool((out[~fin] == -float("inf")).all()) and bool((out[fin] >= 0).all())
    sample = np.array([lo, lo + 1, lo + 4095, lo + 8191, hi - 2, hi - 1], dtype=np.int64)
    ref = parity.oracle_full_scores(dev, wl, sample, ld)
    err = parity.compare_full_scores(out[torch.as_tensor(sample - lo, device="cuda")].cpu().numpy(), ref,
                                     exact=False, what="long_128k")
    print(f"\nlong_128k last chunk: {len(sample)} rows x {ld} pools, max relative error {err:.2e}")
    assert err <= MAX_OBSERVED_REL_ERR
