"""The decode entry point that allocates nothing.

pkv_paged_attention_decode_static_ws serves callers that cannot allocate
device memory where they run attention, such as an engine plugin that may only
use memory it was handed.  Its split-K scratch is a fixed region inside the
library, shared by every call and never cleared.

The calls below go through the C ABI one after another on shapes that take
every schedule the region serves (the work-balanced tensor-core kernel, the
fixed-partition kernel of more than 512 sequences, the CUDA-core kernel with
several partitions in fp32 and at head_dim 64).  The first call runs on a
query full of NaN, so the region starts out holding NaN partials, and every
later call follows one of another shape: a result that read scratch left
over by an earlier call would show.  Each result is compared element by
element with the binary64 oracle (NaN-filled block tails) and with the
workspace entry point.  The file name makes pytest collect it last.
"""
import ctypes
from dataclasses import replace

import pytest
import torch

import pkv_workloads as wl
from conftest import attn_error

pytestmark = pytest.mark.gpu
ATOL_16 = 2e-2
ATOL_32 = 1e-5
STATIC_BYTES = 16 * 1024 * 1024  # PKV_STATIC_WORKSPACE_BYTES


def _call_static(pkv, b, max_ctx, err, q=None):
    q = b.q if q is None else q
    out = torch.empty_like(q)
    c = b.cfg
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = pkv._lib.pkv_paged_attention_decode_static_ws(
        p(out), p(q), p(b.k_cache), p(b.v_cache), p(b.block_tables), b.block_tables.shape[1],
        p(b.context_lens), q.shape[0], c.num_q_heads, c.num_kv_heads, c.head_dim, c.block_size,
        b.k_cache.shape[0], max_ctx, b.scale, pkv._DTYPE[c.dtype], p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pkv.PKV_OK, pkv._lib.pkv_last_error_string()
    return out


# fp32 and head_dim 64 shapes that run the CUDA-core kernel with more than one partition
_F32_GQA = replace(wl.LONG_GQA_8K, name="f32-gqa", dtype=torch.float32, num_q_heads=8, num_kv_heads=2, head_dim=64)
_BF16_D64 = replace(wl.LONG_GQA_8K, name="bf16-d64", num_q_heads=8, num_kv_heads=4, head_dim=64)
_MANY_SEQS = replace(wl.QWEN3_GQA, name="qwen3-520", block_size=16, num_blocks=None)


def _cases():
    g = torch.Generator().manual_seed(5)
    many = torch.randint(1, 601, (520,), generator=g).tolist()
    return [
        (wl.LONG_GQA_8K, [8192, 3000, 1, 5000], 8192),                      # work-balanced, split units
        (_F32_GQA, [3000, 1, 700, 2500], 3000),                              # CUDA-core, fp32, 12 partitions
        (wl.QWEN3_GQA, [300, 7000, 256, 4100, 8000, 19, 0, 2048], 8192),     # work-balanced, ragged
        (_MANY_SEQS, many, 600),                                             # > 512 sequences: fixed partitions
        (_BF16_D64, [4000, 17, 2100], 4000),                                 # CUDA-core, bf16, head_dim 64
    ]


def test_static_workspace_matches_oracle_and_workspace_entry_after_other_shapes(pkv, orc, cuda_dev):
    cases = _cases()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    # Leave NaN partials in the region: a call on a NaN query of the first shape.
    cfg0, lens0, max0 = cases[0]
    b0 = wl.decode_batch(cfg0, seed=39, device=cuda_dev, batch=len(lens0), ctx_override=lens0)
    poisoned = _call_static(pkv, b0, max0, err, q=torch.full_like(b0.q, float("nan")))
    torch.cuda.synchronize()
    assert torch.isnan(poisoned.float()).any()
    for rnd in range(2):  # every shape twice, each call after a call of another shape
        for i, (cfg, lens, max_ctx) in enumerate(cases):
            b = wl.decode_batch(cfg, seed=40 + i + 10 * rnd, device=cuda_dev, batch=len(lens), ctx_override=lens,
                                nan_tails=True)
            need = pkv.pkv_paged_attention_decode_workspace_size(len(lens), cfg.num_q_heads, cfg.num_kv_heads,
                                                                 cfg.head_dim, cfg.block_size, max_ctx, cfg.dtype)
            assert 0 < need <= STATIC_BYTES, (cfg.name, need)
            err.zero_()
            got = _call_static(pkv, b, max_ctx, err)
            want = pkv.pkv_paged_attention_decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens,
                                                  b.scale, max_ctx)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, (cfg.name, int(err.item()))
            ref, nerr = orc.paged_attention_decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens,
                                                   b.scale)
            assert nerr == 0
            tol = ATOL_32 if cfg.dtype == torch.float32 else ATOL_16
            assert attn_error(got, ref) <= tol, cfg.name
            assert (got.double() - want.double()).abs().max().item() <= tol, cfg.name


def test_static_workspace_covers_the_long_context_workload(pkv, orc, cuda_dev):
    # 8 x 32768 tokens, Hq 32 / Hkv 8: the largest scratch of the decode workloads
    cfg = wl.LONG_GQA_32K
    need = pkv.pkv_paged_attention_decode_workspace_size(cfg.batch, cfg.num_q_heads, cfg.num_kv_heads,
                                                         cfg.head_dim, cfg.block_size, cfg.ctx_hi, cfg.dtype)
    assert need <= STATIC_BYTES
    b = wl.decode_batch(cfg, seed=47, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    ref, nerr = orc.paged_attention_decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens, b.scale)
    assert nerr == 0
    for _ in range(2):
        got = _call_static(pkv, b, b.max_context_len, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert attn_error(got, ref) <= ATOL_16


def test_static_workspace_rejects_oversized_requests_and_bad_arguments(pkv, cuda_dev):
    L = pkv._lib
    dummy = torch.zeros(64, dtype=torch.int32, device=cuda_dev)
    p = ctypes.c_void_p(dummy.data_ptr())
    # 4096 sequences x 32 heads x a 1M-token bound needs far more than 16 MiB of
    # scratch: rejected before anything is enqueued (the buffers are never read)
    st = L.pkv_paged_attention_decode_static_ws(p, p, p, p, p, 1, p, 4096, 32, 8, 128, 16, 1000, 1 << 20, 1.0,
                                                pkv.PKV_BF16, None, None)
    assert st == pkv.PKV_ERR_WORKSPACE
    assert b"built-in" in L.pkv_last_error_string()
    # argument errors come first, as on the workspace entry point
    st = L.pkv_paged_attention_decode_static_ws(None, None, None, None, None, 1, None, 4096, 32, 8, 128, 16, 1000,
                                                1 << 20, 1.0, pkv.PKV_BF16, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    st = L.pkv_paged_attention_decode_static_ws(p, p, p, p, p, 1, p, 4, 30, 8, 128, 16, 1000, 64, 1.0,
                                                pkv.PKV_BF16, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG  # 30 query heads over 8 KV heads
