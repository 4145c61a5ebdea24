"""Failure detection on the GPU without a fault: the bounded pipeline wait of
the attention kernels, run on a barrier that nothing completes, ends at its
limit and reports PKV_ERRBIT_TIMEOUT through the error flag; the context stays
usable and the next decode call is exact against the oracle."""
import time

import pytest
import torch

import pkv_workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_sets_the_timeout_bit(pkv, orc, cuda_dev):
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pkv.pkv_selftest_wait_timeout(err, 20000)  # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == pkv.ERRBIT_TIMEOUT
    assert 0.015 <= elapsed < 2.0
    # the context is still usable: a decode call right after is exact
    batch = wl.decode_batch(wl.LONG_GQA_8K, seed=8, device=cuda_dev, batch=3, ctx_override=[700, 33, 1500])
    err.zero_()
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, 1500, err_flag=err)
    ref, nerr = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                           batch.context_lens, batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert (out.cpu().double() - ref).abs().max().item() <= 2e-2
