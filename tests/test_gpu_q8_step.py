"""GPU parity of the 8-bit (E4M3 and int8) caches beyond the one-launch
schedule: more than 512 sequences per call (consecutive work-balanced launches
over groups of sequences), and the fused decode step
(pkv_paged_attention_decode_append_fp8 / _int8) that encodes every sequence's
new K/V row under the block's existing scale into position ctx - 1 and then
attends over the whole context.

Against the oracle, composed the way "Walk the Shapes First" runs a decode
step: the slot of position ctx - 1 (compute_slot_mapping), the 8-bit store of
the new row there (store_kvcache_fp8 / _int8), decode attention over the
codes.  Codes bit-exact, attention within 2e-2 absolute of binary64.
"""
import pytest
import torch

import pkv_workloads as wl
from conftest import attn_error

pytestmark = pytest.mark.gpu

ATOL_16 = 2e-2


def _codes(pkv, fmt, batch):
    quant = getattr(pkv, "pkv_quantize_kvcache_" + fmt)
    kq, ks = quant(batch.k_cache)
    vq, vs = quant(batch.v_cache)
    return kq, ks, vq, vs


def _oracle_q8_step(orc, fmt, batch, kq, ks, vq, vs, key, value):
    """Slot of position ctx - 1, 8-bit store there, attention (CPU copies)."""
    cl = batch.context_lens.cpu()
    keep = (cl > 0).nonzero().reshape(-1)
    bt = batch.block_tables.cpu()
    nb, bs = kq.shape[0], kq.shape[1]
    slots, e1 = orc.compute_slot_mapping(bt[keep], cl[keep] - 1, cl[keep], bs, nb)
    store = getattr(orc, "store_kvcache_" + fmt)
    kc, vc, e2 = store(key.cpu()[keep], value.cpu()[keep], kq.cpu(), vq.cpu(), ks.cpu(), vs.cpu(), slots)
    attend = getattr(orc, "paged_attention_decode_" + fmt)
    out, e3 = attend(batch.q, kc, vc, ks, vs, bt, cl, batch.scale)
    return out, kc, vc, e1 + e2 + e3


def _fused(pkv, fmt, batch, kq, ks, vq, vs, key, value, max_ctx, err):
    fn = getattr(pkv, "pkv_paged_attention_decode_append_" + fmt)
    return fn(batch.q, key, value, kq, vq, ks, vs, batch.block_tables, batch.context_lens, batch.scale, max_ctx,
              err_flag=err)


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_decode_q8_more_than_512_sequences(pkv, orc, cuda_dev, fmt):
    """1100 sequences: three launches of about 367, one workspace reused in
    stream order; NaN in every unused block tail."""
    g = torch.Generator().manual_seed(90)
    B = 1100
    lens = torch.randint(1, 300, (B,), generator=g)
    lens[:6] = torch.tensor([3000, 1234, 16, 17, 0, 2049])
    lens[600:603] = torch.tensor([2500, 0, 1])  # long and empty sequences in a later group too
    cfg = wl.DecodeConfig("t", torch.bfloat16, 16, 8, 128, 16, B, 1, 3000, None)
    batch = wl.decode_batch(cfg, seed=91, device=cuda_dev, ctx_override=lens.tolist(), nan_tails=True)
    kq, ks, vq, vs = _codes(pkv, fmt, batch)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = getattr(pkv, "pkv_paged_attention_decode_" + fmt)(batch.q, kq, vq, ks, vs, batch.block_tables,
                                                             batch.context_lens, batch.scale, 3000, err_flag=err)
    ref, nerr = getattr(orc, "paged_attention_decode_" + fmt)(batch.q, kq, vq, ks, vs, batch.block_tables,
                                                              batch.context_lens, batch.scale)
    assert nerr == 0 and int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert attn_error(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[4]) == 0 and torch.count_nonzero(out[601]) == 0


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (8, 1), (4, 2), (64, 8)])
@pytest.mark.parametrize("bs", [16, 256])
def test_fused_step_q8_matches_oracle(pkv, orc, cuda_dev, fmt, dtype, Hq, Hkv, bs):
    lens = [0, 1, 15, 16, 17, 100, 1000, 2100]
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, len(lens), 1, 2100, 400)
    batch = wl.decode_batch(cfg, seed=2 * Hq + Hkv + bs, device=cuda_dev, ctx_override=lens, nan_tails=True)
    kq, ks, vq, vs = _codes(pkv, fmt, batch)
    # new rows: some beyond the block's range (saturate / clamp); for int8 one
    # NaN, which encodes as 0 (an E4M3 cache would keep it as NaN)
    g = torch.Generator().manual_seed(Hq + bs)
    key = (torch.randn(len(lens), Hkv, 128, generator=g) * 3).to(dtype)
    value = torch.randn(len(lens), Hkv, 128, generator=g).to(dtype)
    if fmt == "int8":
        key[3, 0, 5] = float("nan")
    key, value = key.to(cuda_dev), value.to(cuda_dev)
    ref, kr, vr, nerr = _oracle_q8_step(orc, fmt, batch, kq, ks, vq, vs, key, value)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _fused(pkv, fmt, batch, kq, ks, vq, vs, key, value, 2100, err)
    torch.cuda.synchronize()
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(kq.cpu(), kr) and torch.equal(vq.cpu(), vr)
    assert attn_error(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[0]) == 0


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_fused_step_q8_bad_block_and_many_sequences(pkv, orc, cuda_dev, fmt):
    """700 sequences (two launches) with one table entry out of range at the
    block that holds position ctx - 1: that sequence's append is skipped and
    its block counts as masked (PKV_ERRBIT_BLOCK_RANGE), as in the oracle."""
    g = torch.Generator().manual_seed(93)
    B = 700
    lens = torch.randint(1, 200, (B,), generator=g)
    lens[:3] = torch.tensor([1500, 33, 0])
    lens[650] = 900
    cfg = wl.DecodeConfig("t", torch.bfloat16, 8, 4, 128, 16, B, 1, 1500, None)
    batch = wl.decode_batch(cfg, seed=94, device=cuda_dev, ctx_override=lens.tolist(), nan_tails=True)
    kq, ks, vq, vs = _codes(pkv, fmt, batch)
    bt = batch.block_tables.clone()
    bt[650, (900 - 1) // 16] = 10 ** 6  # the block of position ctx - 1 of sequence 650
    batch.block_tables = bt
    key = torch.randn(B, 4, 128, generator=g).to(torch.bfloat16).to(cuda_dev)
    value = torch.randn(B, 4, 128, generator=g).to(torch.bfloat16).to(cuda_dev)
    ref, kr, vr, nerr = _oracle_q8_step(orc, fmt, batch, kq, ks, vq, vs, key, value)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _fused(pkv, fmt, batch, kq, ks, vq, vs, key, value, 1500, err)
    torch.cuda.synchronize()
    assert nerr >= 1 and int(err.item()) == pkv.ERRBIT_BLOCK_RANGE
    assert torch.equal(kq.cpu(), kr) and torch.equal(vq.cpu(), vr)
    assert attn_error(out, ref) <= ATOL_16


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
@pytest.mark.parametrize("name", ["long-gqa-8k-bf16", "qwen3-0.6b-gqa-bf16"])
def test_full_size_fused_step_q8(pkv, orc, cuda_dev, fmt, name):
    """The workload's decode step over its quantized caches, the whole batch
    against the oracle (codes of every block, every output row)."""
    cfg = wl.CONFIGS[name]
    batch = wl.decode_batch(cfg, seed=95, device=cuda_dev, nan_tails=True)
    kq, ks, vq, vs = _codes(pkv, fmt, batch)
    ref, kr, vr, nerr = _oracle_q8_step(orc, fmt, batch, kq, ks, vq, vs, batch.new_key, batch.new_value)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _fused(pkv, fmt, batch, kq, ks, vq, vs, batch.new_key, batch.new_value, batch.max_context_len, err)
    torch.cuda.synchronize()
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(kq.cpu(), kr) and torch.equal(vq.cpu(), vr)
    assert not torch.isnan(out).any()
    assert attn_error(out, ref) <= ATOL_16
