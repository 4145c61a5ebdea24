"""GPU parity of the int8 cache path against the oracle: quantization and the
slot-mapping store bit-exact (codes and scales), decode attention over the
codes within the bar of the 16-bit path (2e-2 absolute against binary64 on the
dequantized cache).  Scheme ("Block-Paged KV Cache", Quantization
compatibility; symmetric reading): one scale per (block, KV head), max|x| / 127,
codes round-half-even clamped to +-127, NaN -> 0."""
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
def test_quantize_int8_matches_oracle(pkv, orc, cuda_dev, dtype, nb, bs, H, d):
    """Vector and pair kernels (as for E4M3); every code, the NaN's included, is
    the oracle's."""
    g = torch.Generator().manual_seed(60 + d)
    cache = torch.randn(nb, bs, H, d, generator=g) * torch.logspace(-3, 3, nb)[:, None, None, None]
    cache[3, :, H - 1] = 0             # an all-zero (block, head): scale 0, codes 0
    cache[5, 7, 1, 9] = float("nan")   # ignored by the max, stored as 0
    cache[6, 2, 0, 4] = -cache[6].abs().max() * 1.0  # the extreme itself: code -127
    cache = cache.to(dtype)
    codes, scales = pkv.pkv_quantize_kvcache_int8(cache.to(cuda_dev))
    want_codes, want_scales = orc.quantize_kvcache_int8(cache)
    assert codes.dtype == torch.int8
    assert torch.equal(scales.cpu(), want_scales)
    assert torch.equal(codes.cpu(), want_codes)
    assert int(codes[5, 7, 1, 9]) == 0 and int(codes[6, 2, 0, 4]) == -127


def test_quantize_int8_ties_round_to_even(pkv, orc, cuda_dev):
    """Values whose quotient by the scale lands on k + 1/2: with max = 127 the
    scale is exactly 1, so x = k + 0.5 is a tie (fp32 cache, exact)."""
    x = torch.zeros(1, 16, 1, 16, dtype=torch.float32)
    x[0, 0, 0, 0] = 127.0
    ties = torch.tensor([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5, 3.5, 4.5, -3.5, 100.5, 101.5, -7.5, 8.5])
    x[0, 1, 0, :15] = ties
    codes, scales = pkv.pkv_quantize_kvcache_int8(x.to(cuda_dev))
    assert float(scales[0, 0]) == 1.0
    got = codes.cpu()[0, 1, 0, :15].tolist()
    assert got == [0, 2, 2, 0, -2, -2, 126, -126, 4, 4, -4, 100, 102, -8, 8]
    want, _ = orc.quantize_kvcache_int8(x)
    assert torch.equal(codes.cpu(), want)


def test_store_int8_matches_oracle(pkv, orc, cuda_dev):
    g = torch.Generator().manual_seed(61)
    nb, bs, H, d = 12, 16, 8, 128
    base = torch.randn(nb, bs, H, d, generator=g).to(torch.bfloat16)
    kc, ks = orc.quantize_kvcache_int8(base)
    vc, vs = orc.quantize_kvcache_int8(base * 2)
    ks[4, 3] = 0.0  # a zero scale stores 0
    n = 40
    key = (torch.randn(n, H, d, generator=g) * 3).to(torch.bfloat16)  # some beyond 127 * s: clamp
    value = torch.randn(n, H, d, generator=g).to(torch.bfloat16)
    value[9, 2, 5] = float("nan")  # stored as 0
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    slots[5] = -1
    slots[6] = nb * bs + 3  # out of range: skipped, PKV_ERRBIT_SLOT_RANGE
    taken = set(slots.tolist())
    slots[7] = next(r for r in range(4 * bs, 5 * bs) if r not in taken)  # block 4; slots stay distinct
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kd, vd = kc.to(cuda_dev), vc.to(cuda_dev)
    pkv.pkv_store_kvcache_int8(key.to(cuda_dev), value.to(cuda_dev), kd, vd, ks.to(cuda_dev), vs.to(cuda_dev),
                               slots.to(cuda_dev), err_flag=err)
    wk, wv, nerr = orc.store_kvcache_int8(key, value, kc, vc, ks, vs, slots)
    assert nerr == 1 and int(err.item()) == pkv.ERRBIT_SLOT_RANGE
    assert torch.equal(kd.cpu(), wk) and torch.equal(vd.cpu(), wv)
    assert (wk.abs() == 127).any()  # the clamp was exercised


def _int8_case(pkv, cuda_dev, dtype, Hq, Hkv, bs, lens, seed, nan_tails=True):
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, len(lens), 1, max(lens), None)
    batch = wl.decode_batch(cfg, seed=seed, device=cuda_dev, ctx_override=lens, nan_tails=nan_tails)
    kq, ks = pkv.pkv_quantize_kvcache_int8(batch.k_cache)
    vq, vs = pkv.pkv_quantize_kvcache_int8(batch.v_cache)
    return batch, kq, ks, vq, vs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (8, 1), (4, 2), (64, 8)])
@pytest.mark.parametrize("bs", [16, 256])
def test_decode_int8_matches_oracle(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs):
    lens = [0, 1, 15, 16, 17, 100, 1000, 2100]
    batch, kq, ks, vq, vs = _int8_case(pkv, cuda_dev, dtype, Hq, Hkv, bs, lens, seed=Hq + Hkv + bs + 1)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                              batch.scale, max(lens), err_flag=err)
    ref, nerr = orc.paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                                batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[0]) == 0


def test_decode_int8_every_byte_value(pkv, orc, cuda_dev):
    """Caches of raw random bytes, -128 included (a code the encoder never
    writes but a caller may): the widening to f16 is exact for all 256."""
    g = torch.Generator().manual_seed(62)
    B, Hq, Hkv, d, bs, nb = 6, 16, 8, 128, 16, 96
    kq = torch.randint(-128, 128, (nb, bs, Hkv, d), generator=g, dtype=torch.int8)
    vq = torch.randint(-128, 128, (nb, bs, Hkv, d), generator=g, dtype=torch.int8)
    ks = torch.rand(nb, Hkv, generator=g) * 0.02
    vs = torch.rand(nb, Hkv, generator=g) * 0.05
    lens = torch.tensor([1, 16, 33, 250, 700, 1500], dtype=torch.int32)
    bt = torch.randperm(nb, generator=g)[:96].to(torch.int32).reshape(1, 96).repeat(B, 1)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    scale = d ** -0.5
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_int8(q.to(cuda_dev), kq.to(cuda_dev), vq.to(cuda_dev), ks.to(cuda_dev),
                                              vs.to(cuda_dev), bt.to(cuda_dev), lens.to(cuda_dev), scale, 1500,
                                              err_flag=err)
    ref, nerr = orc.paged_attention_decode_int8(q, kq, vq, ks, vs, bt, lens, scale)
    assert nerr == 0 and int(err.item()) == 0
    assert _max_err(out, ref) <= ATOL_16


@pytest.mark.parametrize("Hq,Hkv,bs,ctx,B", [(32, 8, 16, 3000, 3), (8, 8, 256, 40, 3), (4, 1, 16, 1, 7),
                                            (16, 8, 16, 700, 100)])
def test_decode_int8_equal_lengths(pkv, orc, cuda_dev, Hq, Hkv, bs, ctx, B):
    """Every sequence at max_ctx (the early-issue case) over int8 caches."""
    batch, kq, ks, vq, vs = _int8_case(pkv, cuda_dev, torch.bfloat16, Hq, Hkv, bs, [ctx] * B, seed=ctx + B + 1)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                              batch.scale, ctx, err_flag=err)
    ref, nerr = orc.paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                                batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert _max_err(out, ref) <= ATOL_16


def test_decode_int8_peaky_and_split_invariance(pkv, orc, cuda_dev):
    lens = [5000, 777, 4096, 1]
    cfg = wl.LONG_GQA_8K
    batch = wl.decode_batch(cfg, seed=63, device=cuda_dev, batch=4, ctx_override=lens, q_gain=8.0, nan_tails=True)
    kq, ks = pkv.pkv_quantize_kvcache_int8(batch.k_cache)
    vq, vs = pkv.pkv_quantize_kvcache_int8(batch.v_cache)
    ref, _ = orc.paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                             batch.scale)
    full = pkv.pkv_paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                               batch.scale, 5000)
    assert _max_err(full, ref) <= ATOL_16
    for b in range(4):
        one = pkv.pkv_paged_attention_decode_int8(batch.q[b:b + 1].contiguous(), kq, vq, ks, vs,
                                                  batch.block_tables[b:b + 1].contiguous(),
                                                  batch.context_lens[b:b + 1].contiguous(), batch.scale, 5000)
        assert _max_err(one[0], ref[b]) <= ATOL_16


def test_decode_int8_bad_block_and_unsupported_shapes(pkv, orc, cuda_dev):
    batch, kq, ks, vq, vs = _int8_case(pkv, cuda_dev, torch.bfloat16, 16, 8, 16, [300, 600, 0, 50], seed=64)
    bt = batch.block_tables.clone()
    bt[0, 3] = 10_000
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_int8(batch.q, kq, vq, ks, vs, bt, batch.context_lens, batch.scale, 600,
                                              err_flag=err)
    ref, nerr = orc.paged_attention_decode_int8(batch.q, kq, vq, ks, vs, bt, batch.context_lens, batch.scale)
    assert nerr == 1 and int(err.item()) == pkv.ERRBIT_BLOCK_RANGE
    assert _max_err(out, ref) <= ATOL_16
    q64 = torch.zeros(4, 16, 64, dtype=torch.bfloat16, device=cuda_dev)
    k64 = torch.zeros(8, 16, 8, 64, dtype=torch.int8, device=cuda_dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_attention_decode_int8(q64, k64, k64, ks[:8], vs[:8], batch.block_tables, batch.context_lens,
                                            0.1, 600)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["llama2-7b-layer-fp16", "long-gqa-8k-bf16"])
def test_full_size_decode_int8(pkv, orc, cuda_dev, name):
    """The workload quantized on the GPU: codes and scales of every block
    against the oracle, then attention of every sequence against the oracle
    over the GPU's codes."""
    cfg = wl.CONFIGS[name]
    batch = wl.decode_batch(cfg, seed=6, device=cuda_dev, nan_tails=True)
    kq, ks = pkv.pkv_quantize_kvcache_int8(batch.k_cache)
    vq, vs = pkv.pkv_quantize_kvcache_int8(batch.v_cache)
    for src, codes, scales in ((batch.k_cache, kq, ks), (batch.v_cache, vq, vs)):
        wc, wsc = orc.quantize_kvcache_int8(src.cpu())
        assert torch.equal(scales.cpu(), wsc)
        got = codes.cpu()
        finite = ~torch.isnan(src.cpu().float())  # a NaN element's code is checked by the small tests
        assert torch.equal(got[finite], wc[finite])
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                             batch.scale, batch.max_context_len, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()
    ref, nerr = orc.paged_attention_decode_int8(batch.q, kq, vq, ks, vs, batch.block_tables, batch.context_lens,
                                                batch.scale)
    assert nerr == 0
    assert _max_err(out, ref) <= ATOL_16