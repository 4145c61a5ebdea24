"""GPU parity of the causal varlen / chunked prefill attention
(pkv_paged_attention_prefill) against the oracle: max abs error <= 2e-2
(fp16/bf16) against binary64, over caches whose unused rows hold NaN."""
import pytest
import torch

import pkv_workloads as wl
from conftest import attn_error

pytestmark = pytest.mark.gpu

ATOL_16 = 2e-2


def _max_err(out, ref):
    return attn_error(out, ref)


# Launch shapes: every CTA takes two query tiles of one (sequence, KV head), and
# the grid has B * Hkv * ceil(tiles / 2) CTAs for tiles = ceil(max_q_len /
# (128 / G)).  'narrow' gives max_q_len its exact bound (a sequence's last CTA
# may hold a single tile); 'deep' a generous one (many CTAs past a sequence's
# end, which exit at once: a grid many waves deep); 'wide_deep' adds block
# tables of 16k tokens.
WIDE_TABLE_TOKENS = 16384
DEEP_GRID_CTAS = 16 * 2 * 152


def _max_q(mode, mq, B, Hq, Hkv):
    """max_q_len for a test mode: 'narrow' (the exact bound), 'deep' /
    'wide_deep' (a grid of at least DEEP_GRID_CTAS one-tile slots)."""
    if mode == "narrow":
        return mq
    positions = 128 // (Hq // Hkv)
    tiles = -(-DEEP_GRID_CTAS // (B * Hkv))
    return max(mq, tiles * positions)


def _case(dtype, Hq, Hkv, bs, spans, seed, cuda_dev, q_gain=1.0, table_tokens=None):
    """spans: (start, n).  The paged context of sequence b holds start + n tokens
    (unused rows NaN); q holds the n new queries of each sequence.  table_tokens
    widens the block tables (-1 padded) to that many tokens."""
    totals = [s + n for s, n in spans]
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, len(spans), 1, max(totals + [table_tokens or 0]), None)
    batch = wl.decode_batch(cfg, seed=seed, device=cuda_dev, ctx_override=totals, nan_tails=True, nan_unused=True)
    g = torch.Generator().manual_seed(seed + 1)
    ns = [n for _, n in spans]
    q = (torch.randn(sum(ns), Hq, 128, generator=g) * q_gain).to(dtype).to(cuda_dev)
    starts = torch.tensor([s for s, _ in spans], dtype=torch.int32, device=cuda_dev)
    cu = torch.zeros(len(spans) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(ns), 0)
    return batch, q, starts, cu.to(cuda_dev), max(ns)


# (start, new tokens): short and long spans, spans that end on and across
# 128-key block boundaries, and one-token spans
SPANS = [(0, 100), (37, 64), (512, 16), (5, 1), (0, 1), (1000, 200), (16, 48), (127, 130), (128, 128), (0, 257)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (4, 1)])
@pytest.mark.parametrize("bs,mode", [(16, "narrow"), (256, "narrow"), (16, "deep"), (64, "deep"), (256, "deep"),
                                     (16, "wide_deep")])
def test_prefill_matches_oracle(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs, mode):
    batch, q, starts, cu, mq = _case(dtype, Hq, Hkv, bs, SPANS, seed=Hq + Hkv + bs, cuda_dev=cuda_dev,
                                     table_tokens=WIDE_TABLE_TOKENS if mode == "wide_deep" else None)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                          batch.scale, _max_q(mode, mq, len(SPANS), Hq, Hkv), err_flag=err)
    ref, nerr = orc.paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                            batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16


@pytest.mark.parametrize("mode", ["narrow", "deep", "wide_deep"])
def test_prefill_peaky_and_last_row_equals_decode(pkv, orc, cuda_dev, mode):
    """A peaky softmax (q x 8); the last new token of each sequence sees its
    whole context, so its row equals the decode kernel's output there."""
    spans = [(0, 300), (2000, 97), (64, 64)]
    batch, q, starts, cu, mq = _case(torch.bfloat16, 32, 8, 16, spans, seed=70, cuda_dev=cuda_dev, q_gain=8.0,
                                     table_tokens=WIDE_TABLE_TOKENS if mode == "wide_deep" else None)
    out = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                          batch.scale, _max_q(mode, mq, len(spans), 32, 8))
    ref, _ = orc.paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                         batch.scale)
    assert _max_err(out, ref) <= ATOL_16
    last = (cu[1:] - 1).long()
    dec = pkv.pkv_paged_attention_decode(q[last].contiguous(), batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, batch.max_context_len)
    # two kernels, two summation orders: equal up to one ulp of the bf16 output
    # on top of the 1e-2 absolute noise of a sum of unit-size terms
    torch.testing.assert_close(out[last].float(), dec.float(), rtol=2 ** -7, atol=1e-2)


def test_prefill_in_chunks_equals_one_pass(pkv, orc, cuda_dev):
    """Chunked prefill: the same queries split into two calls (positions
    [0, 700) then [700, 1000)) give the rows of one call, and both match the
    oracle's single pass."""
    batch, q, starts, cu, _ = _case(torch.bfloat16, 16, 8, 16, [(0, 1000)], seed=71, cuda_dev=cuda_dev)
    whole = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                            batch.scale, 1000)
    parts = []
    for s, n in ((0, 700), (700, 300)):
        st = torch.tensor([s], dtype=torch.int32, device=cuda_dev)
        c = torch.tensor([0, n], dtype=torch.int32, device=cuda_dev)
        parts.append(pkv.pkv_paged_attention_prefill(q[s:s + n].contiguous(), batch.k_cache, batch.v_cache,
                                                     batch.block_tables, st, c, batch.scale, n))
    # A row's value depends only on its own keys.  The calls cut different query
    # tiles, so P is rounded against different reference maxima: allow one ulp
    # of the bf16 output (2^-7 relative covers it in every binade) on top of
    # the 1e-2 absolute noise of a sum of unit-size terms.
    torch.testing.assert_close(torch.cat(parts).float(), whole.float(), rtol=2 ** -7, atol=1e-2)
    ref, nerr = orc.paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                            batch.scale)
    assert nerr == 0
    assert _max_err(whole, ref) <= ATOL_16 and _max_err(torch.cat(parts), ref) <= ATOL_16


def test_prefill_errors(pkv, orc, cuda_dev):
    spans = [(100, 50), (0, 40)]
    batch, q, starts, cu, mq = _case(torch.bfloat16, 16, 8, 16, spans, seed=72, cuda_dev=cuda_dev)
    bt = batch.block_tables.clone()
    bt[0, 2] = 10_000  # positions 32..47 of sequence 0: dropped
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, bt, starts, cu, batch.scale, mq,
                                          err_flag=err)
    ref, nerr = orc.paged_attention_prefill(q, batch.k_cache, batch.v_cache, bt, starts, cu, batch.scale)
    assert nerr == 1 and int(err.item()) == pkv.ERRBIT_BLOCK_RANGE
    assert _max_err(out, ref) <= ATOL_16
    bad = starts.clone()
    bad[1] = -3  # a negative start: zero rows for that sequence, PKV_ERRBIT_CONTEXT
    err.zero_()
    out = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, bad, cu, batch.scale,
                                          mq, err_flag=err)
    assert int(err.item()) & pkv.ERRBIT_CONTEXT
    assert torch.count_nonzero(out[50:]) == 0
    with pytest.raises(pkv.PkvError) as e:  # head_dim 64: no tensor-core prefill
        pkv.pkv_paged_attention_prefill(torch.zeros(4, 8, 64, dtype=torch.bfloat16, device=cuda_dev),
                                        torch.zeros(8, 16, 8, 64, dtype=torch.bfloat16, device=cuda_dev),
                                        torch.zeros(8, 16, 8, 64, dtype=torch.bfloat16, device=cuda_dev),
                                        batch.block_tables, starts, cu, 0.1, mq)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


def test_prefill_large_sampled_rows(pkv, orc, cuda_dev):
    """A prefill batch of realistic size (32 Hq / 8 Hkv, bf16, 7168 new tokens
    after prefixes of up to 4096): sampled rows against the oracle, each
    recomputed as a one-token span at its position."""
    spans = [(0, 2048), (1024, 1024), (4096, 512), (0, 3584)]
    batch, q, starts, cu, mq = _case(torch.bfloat16, 32, 8, 16, spans, seed=73, cuda_dev=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu,
                                          batch.scale, mq, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and not torch.isnan(out).any()
    picks = []  # (sequence, query index)
    for b, (s, n) in enumerate(spans):
        picks += [(b, 0), (b, n // 2), (b, n - 1)]
    seqs = [b for b, _ in picks]
    rows = [int(cu[b]) + i for b, i in picks]
    st = torch.tensor([spans[b][0] + i for b, i in picks], dtype=torch.int32)
    c1 = torch.arange(len(picks) + 1, dtype=torch.int32)
    ref, nerr = orc.paged_attention_prefill(q.cpu()[rows], batch.k_cache, batch.v_cache,
                                            batch.block_tables.cpu()[seqs], st, c1, batch.scale)
    assert nerr == 0
    assert _max_err(out[torch.tensor(rows, device=cuda_dev)], ref) <= ATOL_16


@pytest.mark.parametrize("mode", ["narrow", "deep"])
def test_prefill_negative_scale(pkv, orc, cuda_dev, mode):
    """A non-positive scale takes the kernel variant that scales each score
    before the maximum (a positive scale is folded into the exponent)."""
    spans = [(0, 100), (300, 70), (17, 1)]
    batch, q, starts, cu, mq = _case(torch.bfloat16, 16, 8, 16, spans, seed=74, cuda_dev=cuda_dev)
    scale = -0.7 * batch.scale
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu, scale,
                                          _max_q(mode, mq, len(spans), 16, 8), err_flag=err)
    ref, nerr = orc.paged_attention_prefill(q, batch.k_cache, batch.v_cache, batch.block_tables, starts, cu, scale)
    assert nerr == 0 and int(err.item()) == 0
    assert _max_err(out, ref) <= ATOL_16
