"""GPU parity of the fp8 (E4M3) cache path against the oracle: quantization
and the slot-mapping store bit-exact (codes and scales), decode attention over
the codes within the bar of the 16-bit path (2e-2 absolute against binary64 on
the dequantized cache)."""
import pytest
import torch

import pkv_workloads as wl
from conftest import attn_error

pytestmark = pytest.mark.gpu

ATOL_16 = 2e-2


def _max_err(out, ref):
    return attn_error(out, ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("nb,bs,H,d", [(24, 16, 8, 128), (10, 16, 4, 72), (10, 16, 3, 36), (7, 32, 2, 128)])
def test_quantize_fp8_matches_oracle(pkv, orc, cuda_dev, dtype, nb, bs, H, d):
    """Vector kernel (16-byte loads, slice in registers) where the slice fits,
    pair kernel otherwise (d = 36, 32-token blocks, fp32 rows of 128)."""
    g = torch.Generator().manual_seed(50 + d)
    cache = torch.randn(nb, bs, H, d, generator=g) * torch.logspace(-3, 3, nb)[:, None, None, None]
    cache[3, :, H - 1] = 0        # an all-zero (block, head): scale 0, codes +0
    cache[5, 7, 1, 9] = float("nan")  # ignored by the max, stored as NaN
    cache = cache.to(dtype)
    codes, scales = pkv.pkv_quantize_kvcache_fp8(cache.to(cuda_dev))
    want_codes, want_scales = orc.quantize_kvcache_fp8(cache)
    assert torch.equal(scales.cpu(), want_scales)
    got = codes.cpu()
    nan = torch.zeros_like(got, dtype=torch.bool)
    nan[5, 7, 1, 9] = True
    assert (got[nan] & 0x7F).item() == 0x7F  # a NaN code
    assert torch.equal(got[~nan], want_codes[~nan])


def test_store_fp8_matches_oracle(pkv, orc, cuda_dev):
    g = torch.Generator().manual_seed(51)
    nb, bs, H, d = 12, 16, 8, 128
    base = torch.randn(nb, bs, H, d, generator=g).to(torch.bfloat16)
    kc, ks = orc.quantize_kvcache_fp8(base)
    vc, vs = orc.quantize_kvcache_fp8(base * 2)
    ks[4, 3] = 0.0  # a zero scale stores +0
    n = 40
    key = (torch.randn(n, H, d, generator=g) * 3).to(torch.bfloat16)  # some beyond 448 * s: saturate
    value = torch.randn(n, H, d, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    slots[5] = -1
    slots[6] = nb * bs + 3  # out of range: skipped, PKV_ERRBIT_SLOT_RANGE
    taken = set(slots.tolist())
    slots[7] = next(r for r in range(4 * bs, 5 * bs) if r not in taken)  # block 4; slots stay distinct
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kd, vd = kc.to(cuda_dev), vc.to(cuda_dev)
    pkv.pkv_store_kvcache_fp8(key.to(cuda_dev), value.to(cuda_dev), kd, vd, ks.to(cuda_dev), vs.to(cuda_dev),
                              slots.to(cuda_dev), err_flag=err)
    wk, wv, nerr = orc.store_kvcache_fp8(key, value, kc, vc, ks, vs, slots)
    assert nerr == 1 and int(err.item()) == pkv.ERRBIT_SLOT_RANGE
    assert torch.equal(kd.cpu(), wk) and torch.equal(vd.cpu(), wv)


def _fp8_case(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs, lens, seed, nan_tails=True):
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, len(lens), 1, max(lens), None)
    batch = wl.decode_batch(cfg, seed=seed, device=cuda_dev, ctx_override=lens, nan_tails=nan_tails)
    kq, ks = pkv.pkv_quantize_kvcache_fp8(batch.k_cache)
    vq, vs = pkv.pkv_quantize_kvcache_fp8(batch.v_cache)
    return batch, kq, ks, vq, vs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (8, 1), (4, 2), (64, 8)])
@pytest.mark.parametrize("bs", [16, 256])
def test_decode_fp8_matches_oracle(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs):
    lens = [0, 1, 15, 16, 17, 100, 1000, 2100]
    batch, kq, ks, vq, vs = _fp8_case(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs, lens, seed=Hq + Hkv + bs)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                             batch.scale, max(lens), err_flag=err)
    ref, nerr = orc.paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                               batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[0]) == 0


@pytest.mark.parametrize("Hq,Hkv,bs,ctx,B", [(32, 8, 16, 3000, 3), (8, 8, 256, 40, 3), (4, 1, 16, 1, 7),
                                            (16, 8, 16, 700, 100)])
def test_decode_fp8_equal_lengths(pkv, orc, cuda_dev, Hq, Hkv, bs, ctx, B):
    """Every sequence at max_ctx (the early-issue case) over E4M3 caches."""
    batch, kq, ks, vq, vs = _fp8_case(pkv, orc, cuda_dev, torch.bfloat16, Hq, Hkv, bs, [ctx] * B, seed=ctx + B)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                             batch.scale, ctx, err_flag=err)
    ref, nerr = orc.paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                               batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert _max_err(out, ref) <= ATOL_16


def test_decode_fp8_peaky_and_split_invariance(pkv, orc, cuda_dev):
    """A peaky softmax (q x 8) over long sequences: alone (spread over every
    CTA) and in a batch, against the oracle."""
    lens = [5000, 777, 4096, 1]
    cfg = wl.LONG_GQA_8K
    batch = wl.decode_batch(cfg, seed=52, device=cuda_dev, batch=4, ctx_override=lens, q_gain=8.0, nan_tails=True)
    kq, ks = pkv.pkv_quantize_kvcache_fp8(batch.k_cache)
    vq, vs = pkv.pkv_quantize_kvcache_fp8(batch.v_cache)
    ref, _ = orc.paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                            batch.scale)
    full = pkv.pkv_paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                              batch.scale, 5000)
    assert _max_err(full, ref) <= ATOL_16
    for b in range(4):
        one = pkv.pkv_paged_attention_decode_fp8(batch.q[b:b + 1].contiguous(), kq, vq, ks, vs,
                                                 batch.block_tables[b:b + 1].contiguous(),
                                                 batch.context_lens[b:b + 1].contiguous(), batch.scale, 5000)
        assert _max_err(one[0], ref[b]) <= ATOL_16


def test_decode_fp8_bad_block_and_unsupported_shapes(pkv, orc, cuda_dev):
    batch, kq, ks, vq, vs = _fp8_case(pkv, orc, cuda_dev, torch.bfloat16, 16, 8, 16, [300, 600, 0, 50], seed=53)
    bt = batch.block_tables.clone()
    bt[0, 3] = 10_000
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, bt, batch.context_lens, batch.scale, 600,
                                             err_flag=err)
    ref, nerr = orc.paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, bt, batch.context_lens, batch.scale)
    assert nerr == 1 and int(err.item()) == pkv.ERRBIT_BLOCK_RANGE
    assert _max_err(out, ref) <= ATOL_16
    # shapes outside the tensor-core work-balanced path are refused before any launch
    q64 = torch.zeros(4, 16, 64, dtype=torch.bfloat16, device=cuda_dev)
    k64 = torch.zeros(8, 16, 8, 64, dtype=torch.uint8, device=cuda_dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_attention_decode_fp8(q64, k64, k64, ks[:8], vs[:8], batch.block_tables, batch.context_lens,
                                           0.1, 600)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["llama2-7b-layer-fp16", "long-gqa-8k-bf16"])
def test_full_size_decode_fp8(pkv, orc, cuda_dev, name):
    """The workload quantized on the GPU: codes and scales of every block
    against the oracle, then attention of every sequence against the oracle
    over the GPU's codes."""
    cfg = wl.CONFIGS[name]
    batch = wl.decode_batch(cfg, seed=4, device=cuda_dev, nan_tails=True)
    kq, ks = pkv.pkv_quantize_kvcache_fp8(batch.k_cache)
    vq, vs = pkv.pkv_quantize_kvcache_fp8(batch.v_cache)
    for src, codes, scales in ((batch.k_cache, kq, ks), (batch.v_cache, vq, vs)):
        wc, wsc = orc.quantize_kvcache_fp8(src.cpu())
        assert torch.equal(scales.cpu(), wsc)
        got = codes.cpu()
        finite = ~torch.isnan(src.cpu().float())  # a NaN element's code is checked by the small tests
        assert torch.equal(got[finite], wc[finite])
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                             batch.scale, batch.max_context_len, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()
    ref, nerr = orc.paged_attention_decode_fp8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                                batch.scale)
    assert nerr == 0
    assert _max_err(out, ref) <= ATOL_16