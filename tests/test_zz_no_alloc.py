"""The decode entry point that allocates nothing.

pkv_paged_attention_decode_static_ws serves callers that cannot allocate
device memory where they run attention, such as an engine plugin that may only
use memory it was handed.  Its split-K scratch is a fixed region inside the
library.  Called through the C ABI, two calls in a row with different shapes
must match the workspace entry point within the attention tolerance.  The
second call checks that scratch left over by the first does not leak into the
result.  The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import pkv_workloads as wl

pytestmark = pytest.mark.gpu
ATOL_16 = 2e-2


def _call_static(pkv, b, max_ctx, err):
    out = torch.empty_like(b.q)
    c = b.cfg
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = pkv._lib.pkv_paged_attention_decode_static_ws(
        p(out), p(b.q), p(b.k_cache), p(b.v_cache), p(b.block_tables), b.block_tables.shape[1],
        p(b.context_lens), b.q.shape[0], c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size,
        b.k_cache.shape[0], max_ctx, b.scale, pkv._DTYPE[c.dtype], p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pkv.PKV_OK, pkv._lib.pkv_last_error_string()
    return out


def test_static_workspace_matches_workspace_entry_point_twice(pkv, cuda_dev):
    cases = [
        (wl.LONG_GQA_8K, [8192, 3000, 1, 5000], 8192),                 # several partitions per sequence
        (wl.QWEN3_GQA, [300, 7000, 256, 4100, 8000, 19, 0, 2048], 8192),  # different shape, ragged
    ]
    for i, (cfg, lens, max_ctx) in enumerate(cases):
        b = wl.decode_batch(cfg, seed=40 + i, device=cuda_dev, batch=len(lens), ctx_override=lens, nan_tails=True)
        need = pkv.pkv_paged_attention_decode_workspace_size(len(lens), cfg.num_q_heads, cfg.num_kv_heads,
                                                             cfg.head_dim, cfg.block_size, max_ctx, cfg.dtype)
        assert 0 < need <= 16 * 1024 * 1024
        err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
        got = _call_static(pkv, b, max_ctx, err)
        want = pkv.pkv_paged_attention_decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens,
                                              b.scale, max_ctx)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert (got.float() - want.float()).abs().max().item() <= ATOL_16


def test_static_workspace_rejects_oversized_requests(pkv, cuda_dev):
    # 4096 sequences x 32 heads x a 1M-token bound needs far more than 16 MiB of scratch
    st = pkv._lib.pkv_paged_attention_decode_static_ws(None, None, None, None, None, 1, None, 4096, 32, 8, 128,
                                                       16, 1000, 1 << 20, 1.0, pkv.PKV_BF16, None, None)
    assert st == pkv.PKV_ERR_WORKSPACE
    assert b"built-in" in pkv._lib.pkv_last_error_string()
