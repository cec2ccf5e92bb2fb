"""The workspace-free entry point, kpool_select_static_scratch.

It exists for callers that cannot allocate device memory (a plugin inside a
framework that owns every device allocation, a real-time path that must not hit
cudaMalloc): it runs the same kernels as kpool_select with its scratch in a
fixed array compiled into the library. Same kernels on the same inputs, so its
outputs must equal kpool_select's bit for bit -- scores included. The array is
shared by every call and keeps the last call's contents, so the GPU tests run
calls of different sizes back to back (a larger batch, then a smaller one, then
a larger one again) and a malformed batch followed by a valid one: nothing a
previous call left in the array may reach a later call's outputs. This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_kpool_gb300 import build as kbuild
from sparse_attention_kpool_gb300 import kpool as K
from sparse_attention_kpool_gb300 import workloads as W


def test_static_scratch_rejects_before_any_gpu_work():
    """Every case here fails host validation, so no kernel sees the fake pointers."""
    kbuild.build()
    lib = K.load()
    P = ctypes.c_void_p
    fake = 0x7F0000000000
    T = 1 << 22  # 4M tokens: the workspace would be ~270 MB, beyond the 48 MiB array
    assert K.kpool_workspace_bytes(T, 1, 32, 128, K.KPOOL_BF16, 4, 2048) > K.KPOOL_STATIC_SCRATCH_BYTES
    st = lib.kpool_select_static_scratch(P(fake), P(fake), P(fake), P(fake), 1, T, 32, 128, K.KPOOL_BF16, 4, 2048,
                                         0.1, P(fake), P(fake), None, None)
    assert st == K.KPOOL_ERR_WORKSPACE
    # a shape the kernels do not implement is reported as such at any size, before capacity
    for t in (64, T):
        assert lib.kpool_select_static_scratch(P(fake), P(fake), P(fake), P(fake), 1, t, 65, 128, K.KPOOL_BF16, 4,
                                               2048, 0.1, P(fake), P(fake), None, None) == K.KPOOL_ERR_UNSUPPORTED
    # invalid arguments likewise, at any size
    for t in (64, T):
        assert lib.kpool_select_static_scratch(P(fake), P(fake), P(fake), P(fake), 1, t, 32, 128, K.KPOOL_BF16, 3,
                                               2048, 0.1, P(fake), P(fake), None, None) == K.KPOOL_ERR_INVALID_ARG
        assert lib.kpool_select_static_scratch(P(fake + 2), P(fake), P(fake), P(fake), 1, t, 32, 128, K.KPOOL_BF16,
                                               4, 2048, 0.1, P(fake), P(fake), None, None) == K.KPOOL_ERR_INVALID_ARG
    # an empty batch is a no-op
    assert lib.kpool_select_static_scratch(None, None, None, None, 0, 0, 32, 128, K.KPOOL_BF16, 4, 2048, 0.1,
                                           None, None, None, None) == K.KPOOL_OK


def _batch(name, seqlens, values, seed):
    wl = W.custom(name, seqlens, 32, 128, 4, 2048, 1.0 / 16 if values == "integer" else 1.0 / np.sqrt(128), "bf16",
                  values, seed, dup_every=8 if values == "integer" else 0)
    return wl, {k: v.cuda() for k, v in W.generate(wl, "cpu").items()}


def _both_paths(wl, dev):
    ref = K.kpool_select(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk, wl.scale,
                         return_scores=True)
    got = K.kpool_select_static_scratch(dev["q"], dev["k"], dev["w"], dev["cu_seqlens"], wl.kpool, wl.index_topk,
                                        wl.scale, return_scores=True)
    torch.cuda.synchronize()
    assert K.kpool_static_scratch_last_device_error() == K.KPOOL_OK
    return [x.cpu().numpy() for x in ref], [x.cpu().numpy() for x in got]


@pytest.mark.gpu
@pytest.mark.parametrize("values", ["integer", "normal"])
def test_static_scratch_equals_workspace_path_across_sizes(values):
    """Large, small, large again, then the first batch once more: each call's ids, tokens and
    scores equal kpool_select's bit for bit (same kernels, same inputs)."""
    kbuild.build()
    K.load()
    seq = [_batch("noalloc_a", (5000, 1200, 7, 9000), values, 71),
           _batch("noalloc_b", (700, 3), values, 72),
           _batch("noalloc_c", (2, 16000), values, 73)]
    seq.append(seq[0])
    for wl, dev in seq:
        ref, got = _both_paths(wl, dev)
        for name, a, b in zip(("pool ids", "token ids", "scores"), ref, got):
            np.testing.assert_array_equal(b, a, err_msg=f"{wl.name}: {name}")


@pytest.mark.gpu
def test_static_scratch_reports_device_errors_and_recovers():
    """Malformed cu_seqlens is found on the device: the error is read back through
    kpool_static_scratch_last_device_error, nothing is written, and the next valid call on
    the same array succeeds with the workspace path's answer."""
    kbuild.build()
    K.load()
    wl, dev = _batch("noalloc_err", (64, 64), "integer", 74)
    T = wl.total_tokens
    for bad in ([0, 100, 90], [1, 64, 128], [0, 64, 127]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        ids = torch.full((T, wl.budget), 777, dtype=torch.int32, device="cuda")
        toks = torch.full((T, wl.width), 777, dtype=torch.int32, device="cuda")
        K.kpool_select_static_scratch(dev["q"], dev["k"], dev["w"], cu, wl.kpool, wl.index_topk, wl.scale,
                                      out_pool_ids=ids, out_token_ids=toks)
        assert K.kpool_static_scratch_last_device_error() == K.KPOOL_ERR_INVALID_ARG
        assert bool((toks == 777).all()) and bool((ids == 777).all())
    ref, got = _both_paths(wl, dev)
    for a, b in zip(ref, got):
        np.testing.assert_array_equal(b, a)
