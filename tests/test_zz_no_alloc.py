"""The workspace-free entry point, kpool_select_static_scratch.

It exists for callers that cannot allocate device memory (a plugin inside a
framework that owns every device allocation, a real-time path that must not hit
cudaMalloc): it runs the same kernels as kpool_select with its scratch in a
fixed array compiled into the library. This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_kpool_gb300 import build as kbuild
from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import workloads as W

TOL_REL = 1e-3  # the score tolerance the parity tests use


def test_static_scratch_rejects_oversized_batches():
    kbuild.build()
    lib = K.load()
    P = ctypes.c_void_p
    fake = 0x7F0000000000
    T = 1 << 22  # 4M tokens: the workspace would be ~270 MB, beyond the 48 MiB array
    assert K.kpool_workspace_bytes(T, 1, 32, 128, K.KPOOL_BF16, 4, 2048) > K.KPOOL_STATIC_SCRATCH_BYTES
    st = lib.kpool_select_static_scratch(P(fake), P(fake), P(fake), P(fake), 1, T, 32, 128, K.KPOOL_BF16, 4, 2048,
                                         0.1, P(fake), P(fake), None, None)
    assert st == K.KPOOL_ERR_WORKSPACE
    assert lib.kpool_select_static_scratch(P(fake), P(fake), P(fake), P(fake), 1, 64, 32, 128, K.KPOOL_BF16, 3,
                                           2048, 0.1, P(fake), P(fake), None, None) == K.KPOOL_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("values", ["integer", "normal"])
def test_static_scratch_matches_workspace_path_twice(values):
    kbuild.build()
    K.load()
    wl = W.custom("noalloc", (5000, 1200, 7), 32, 128, 4, 2048,
                  1.0 / 16 if values == "integer" else 1.0 / np.sqrt(128), "bf16", values, 71,
                  dup_every=8 if values == "integer" else 0)
    dev = {k: v.cuda() for k, v in W.generate(wl, "cpu").items()}
    ref_ids, ref_toks, ref_sc = K.kpool_select(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool,
                                               wl.index_topk, wl.scale, return_scores=True)
    torch.cuda.synchronize()
    ref_ids, ref_toks, ref_sc = ref_ids.cpu().numpy(), ref_toks.cpu().numpy(), ref_sc.cpu().numpy()
    for _ in range(2):  # two calls in a row share (and reuse) the built-in scratch
        ids, toks, sc = K.kpool_select_static_scratch(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool,
                                                      wl.index_topk, wl.scale, return_scores=True)
        torch.cuda.synchronize()
        ids, toks, sc = ids.cpu().numpy(), toks.cpu().numpy(), sc.cpu().numpy()
        np.testing.assert_array_equal(ids, ref_ids)
        np.testing.assert_array_equal(toks, ref_toks)
        valid = ref_ids >= 0
        np.testing.assert_allclose(sc[valid], ref_sc[valid], rtol=TOL_REL, atol=0)
        assert (sc[~valid] == -np.inf).all()
