"""GPU parity of the fused decode step (pkv_paged_attention_decode_append):
append every sequence's new K/V row at position ctx - 1, then attend over the
whole context.  Against the oracle's decode_step (slot mapping + store +
attention in binary64): caches bit-exact, attention within the bars of the
plain decode.  Against the library's own three calls: bit-identical.
"""
import pytest
import torch

import pkv_workloads as wl
from conftest import attn_error

pytestmark = pytest.mark.gpu

ATOL_16 = 2e-2
ATOL_32 = 1e-5


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _max_err(out, ref):
    return attn_error(out, ref)


def _append(pkv, batch, max_ctx, err=None, key=None, value=None):
    return pkv.pkv_paged_attention_decode_append(
        batch.q, batch.new_key if key is None else key, batch.new_value if value is None else value,
        batch.k_cache, batch.v_cache, batch.block_tables, batch.context_lens, batch.scale, max_ctx, err_flag=err)


def _oracle_step(orc, batch, kc, vc):
    return orc.decode_step(batch.q, batch.new_key, batch.new_value, kc, vc, batch.block_tables,
                           batch.context_lens, batch.scale)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (8, 1), (4, 2), (64, 8)])
@pytest.mark.parametrize("bs", [16, 256])
def test_append_fused_matches_oracle_step(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs):
    lens = [0, 1, 15, 16, 17, 100, 1000, 2100]
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, len(lens), 1, 2100, 400)
    batch = wl.decode_batch(cfg, seed=Hq + 3 * Hkv + bs, device=cuda_dev, ctx_override=lens, nan_tails=True,
                            nan_unused=True)
    part, _, fast = pkv.pkv_paged_attention_decode_plan(len(lens), Hq, Hkv, 128, bs, 2100, dtype)
    assert fast and part == 0  # the work-balanced kernel, which appends in place
    kc0, vc0 = batch.k_cache.cpu(), batch.v_cache.cpu()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _append(pkv, batch, 2100, err)
    ref, kr, vr, nerr = _oracle_step(orc, batch, kc0, vc0)
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(_bits(batch.k_cache), _bits(kr)) and torch.equal(_bits(batch.v_cache), _bits(vr))
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[0]) == 0


@pytest.mark.parametrize("Hq,Hkv,bs,ctx,B", [(32, 8, 16, 3000, 3), (16, 8, 16, 300, 5), (4, 1, 16, 1, 7),
                                            (8, 2, 16, 17, 40), (16, 8, 256, 700, 6)])
def test_append_fused_equal_lengths(pkv, orc, cuda_dev, Hq, Hkv, bs, ctx, B):
    """Every sequence at max_ctx (the early-issue case): the stage holding
    position ctx - 1 still appends before its copy, and the step matches the
    oracle."""
    cfg = wl.DecodeConfig("t", torch.bfloat16, Hq, Hkv, 128, bs, B, 1, ctx, None)
    batch = wl.decode_batch(cfg, seed=ctx + 2 * B, device=cuda_dev, ctx_override=[ctx] * B, nan_tails=True,
                            nan_unused=True)
    kc0, vc0 = batch.k_cache.cpu(), batch.v_cache.cpu()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _append(pkv, batch, ctx, err)
    ref, kr, vr, nerr = _oracle_step(orc, batch, kc0, vc0)
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(_bits(batch.k_cache), _bits(kr)) and torch.equal(_bits(batch.v_cache), _bits(vr))
    assert _max_err(out, ref) <= ATOL_16


def test_append_equals_the_three_calls(pkv, orc, cuda_dev):
    """Fused step == slot mapping + store + attention through the library, bit
    for bit, and both equal the oracle's decode step."""
    cfg = wl.LONG_GQA_8K
    lens = [8192, 5000, 17, 1, 4096, 777, 16, 2048]
    a = wl.decode_batch(cfg, seed=21, device=cuda_dev, ctx_override=lens, nan_tails=True)
    b = wl.decode_batch(cfg, seed=21, device=cuda_dev, ctx_override=lens, nan_tails=True)
    kc0, vc0 = a.k_cache.cpu(), a.v_cache.cpu()
    out_fused = _append(pkv, a, 8192)
    nb = b.extra["num_blocks"]
    slots = pkv.pkv_compute_slot_mapping(b.block_tables, b.starts, b.ends, b.cu_new, cfg.block_size, nb,
                                         num_new_tokens=len(lens))
    pkv.pkv_store_kvcache(b.new_key, b.new_value, b.k_cache, b.v_cache, slots)
    out_sep = pkv.pkv_paged_attention_decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens, b.scale,
                                             8192)
    torch.cuda.synchronize()
    assert torch.equal(_bits(a.k_cache), _bits(b.k_cache)) and torch.equal(_bits(a.v_cache), _bits(b.v_cache))
    assert torch.equal(_bits(out_fused), _bits(out_sep))
    ref, kr, vr, nerr = _oracle_step(orc, a, kc0, vc0)
    assert nerr == 0
    assert torch.equal(_bits(a.k_cache), _bits(kr)) and torch.equal(_bits(a.v_cache), _bits(vr))
    assert _max_err(out_fused, ref) <= ATOL_16


@pytest.mark.parametrize("case", ["fixed_partitions", "generic_fp32", "generic_fp16_d64", "unaligned_key"])
def test_append_other_paths(pkv, orc, cuda_dev, case):
    """Where the attention kernel does not append itself, the append kernel
    runs first; the result is the same step."""
    if case == "fixed_partitions":  # more than 512 sequences
        g = torch.Generator().manual_seed(31)
        lens = torch.randint(1, 300, (600,), generator=g).tolist()
        lens[:3] = [2500, 16, 17]
        cfg = wl.DecodeConfig("t", torch.bfloat16, 8, 4, 128, 16, 600, 1, 2500, 12000)
        tol = ATOL_16
    elif case == "generic_fp32":  # the page's shapes
        lens = [1, 4, 11, 6]
        cfg = wl.DecodeConfig("t", torch.float32, 4, 2, 8, 4, 4, 1, 11, 16)
        tol = ATOL_32
    elif case == "generic_fp16_d64":
        lens = [1, 63, 64, 65, 1000]
        cfg = wl.DecodeConfig("t", torch.float16, 8, 2, 64, 16, 5, 1, 1000, 100)
        tol = ATOL_16
    else:  # a key/value buffer that is only 2-byte aligned
        lens = [3000, 1, 999, 16]
        cfg = wl.DecodeConfig("t", torch.bfloat16, 32, 8, 128, 16, 4, 1, 3000, 400)
        tol = ATOL_16
    batch = wl.decode_batch(cfg, seed=32, device=cuda_dev, ctx_override=lens, nan_tails=True)
    key, value = batch.new_key, batch.new_value
    if case == "unaligned_key":
        fk = torch.empty(key.numel() + 1, dtype=key.dtype, device=cuda_dev)
        fv = torch.empty_like(fk)
        key = fk[1:].view(key.shape)
        value = fv[1:].view(value.shape)
        key.copy_(batch.new_key)
        value.copy_(batch.new_value)
        assert key.data_ptr() % 8 != 0
    kc0, vc0 = batch.k_cache.cpu(), batch.v_cache.cpu()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _append(pkv, batch, max(lens), err, key, value)
    ref, kr, vr, nerr = _oracle_step(orc, batch, kc0, vc0)
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(_bits(batch.k_cache), _bits(kr)) and torch.equal(_bits(batch.v_cache), _bits(vr))
    assert _max_err(out, ref) <= tol


def test_append_error_semantics(pkv, orc, cuda_dev):
    cfg = wl.DecodeConfig("t", torch.bfloat16, 16, 8, 128, 16, 4, 1, 600, 200)
    batch = wl.decode_batch(cfg, seed=33, device=cuda_dev, ctx_override=[300, 600, 0, 50])
    # sequence 0's last block (position 299 is in logical block 18) points outside the pool
    batch.block_tables[0, 18] = 10_000
    kc0, vc0 = batch.k_cache.clone(), batch.v_cache.clone()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _append(pkv, batch, 600, err)
    assert int(err.item()) == pkv.ERRBIT_BLOCK_RANGE
    ref, kr, vr, nerr = _oracle_step(orc, batch, kc0, vc0)
    assert nerr >= 1
    assert torch.equal(_bits(batch.k_cache), _bits(kr)) and torch.equal(_bits(batch.v_cache), _bits(vr))
    assert _max_err(out, ref) <= ATOL_16
    # a context longer than the declared bound: no append for it, zero row, PKV_ERRBIT_CONTEXT
    batch2 = wl.decode_batch(cfg, seed=34, device=cuda_dev, ctx_override=[300, 600, 0, 50])
    kc0 = batch2.k_cache.clone()
    err.zero_()
    out = _append(pkv, batch2, 400, err)
    assert int(err.item()) & pkv.ERRBIT_CONTEXT
    assert torch.count_nonzero(out[1]) == 0
    p = 599
    blk = int(batch2.block_tables[1, p // 16])
    assert torch.equal(_bits(batch2.k_cache[blk, p % 16]), _bits(kc0[blk, p % 16]))
    for b, n in ((0, 300), (3, 50)):  # the valid ones were appended
        blk = int(batch2.block_tables[b, (n - 1) // 16])
        assert torch.equal(_bits(batch2.k_cache[blk, (n - 1) % 16]), _bits(batch2.new_key[b]))


@pytest.mark.parametrize("name", ["llama2-7b-layer-fp16", "long-gqa-8k-bf16"])
def test_full_size_append_step(pkv, orc, cuda_dev, name):
    """The fused step at full size: caches bit-exact against the oracle's
    store, and the attention of a sample of sequences against the oracle."""
    cfg = wl.CONFIGS[name]
    batch = wl.decode_batch(cfg, seed=3, device=cuda_dev, nan_tails=True)
    kc0, vc0 = batch.k_cache.cpu(), batch.v_cache.cpu()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = _append(pkv, batch, batch.max_context_len, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slots, _ = orc.compute_slot_mapping(batch.block_tables, batch.starts, batch.ends, cfg.block_size,
                                        batch.extra["num_blocks"])
    kr, vr, _ = orc.store_kvcache(batch.new_key, batch.new_value, kc0, vc0, slots)
    del kc0, vc0
    assert torch.equal(_bits(batch.k_cache), _bits(kr)) and torch.equal(_bits(batch.v_cache), _bits(vr))
    sample = [0, cfg.batch // 2, cfg.batch - 1]
    idx = torch.tensor(sample)
    ref, _ = orc.paged_attention_decode(batch.q.cpu()[idx], kr, vr, batch.block_tables.cpu()[idx],
                                        batch.context_lens.cpu()[idx], batch.scale)
    assert _max_err(out[idx.to(cuda_dev)], ref) <= ATOL_16


def test_allocator_driven_decode_steps(pkv, orc, cuda_dev):
    """Several decode steps of a changing batch: the host allocator hands out
    the blocks (a new one exactly when a length becomes 1 mod 16), sequences
    finish and new ones are admitted into freed blocks, and every step runs the
    fused append + attention.  Each step's caches match the oracle's decode
    step bit for bit, the new rows sit at the allocator's slots, and the
    attention is within the bar."""
    g = torch.Generator().manual_seed(40)
    nb, bs, Hq, Hkv, d, dtype = 160, 16, 32, 8, 128, torch.bfloat16
    a = pkv.pkv_allocator_create(nb, bs)
    kc = torch.randn(nb, bs, Hkv, d, generator=g).to(dtype).to(cuda_dev)
    vc = torch.randn(nb, bs, Hkv, d, generator=g).to(dtype).to(cuda_dev)
    live, next_id = [], 0
    for n in (300, 17, 16, 1, 900, 64):
        pkv.pkv_allocator_add_sequence(a, next_id, n)
        live.append(next_id)
        next_id += 1
    for step in range(6):
        if step in (2, 4):  # one sequence finishes, a new one is admitted
            pkv.pkv_allocator_release(a, live.pop(1))
            pkv.pkv_allocator_add_sequence(a, next_id, 40 + 100 * step)
            live.append(next_id)
            next_id += 1
        slots = [pkv.pkv_allocator_append(a, s)[0] for s in live]
        assert pkv.pkv_allocator_check(a) == 0
        rows = [pkv.pkv_allocator_block_table(a, s, 64) for s in live]
        tables = torch.tensor([r[0] for r in rows], dtype=torch.int32)
        lens = torch.tensor([r[1] for r in rows], dtype=torch.int32)
        B = len(live)
        q = torch.randn(B, Hq, d, generator=g).to(dtype)
        key = torch.randn(B, Hkv, d, generator=g).to(dtype)
        value = torch.randn(B, Hkv, d, generator=g).to(dtype)
        kc0, vc0 = kc.cpu(), vc.cpu()
        err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
        out = pkv.pkv_paged_attention_decode_append(q.to(cuda_dev), key.to(cuda_dev), value.to(cuda_dev), kc, vc,
                                                    tables.to(cuda_dev), lens.to(cuda_dev), d ** -0.5,
                                                    int(lens.max()), err_flag=err)
        ref, kr, vr, nerr = orc.decode_step(q, key, value, kc0, vc0, tables, lens, d ** -0.5)
        assert nerr == 0 and int(err.item()) == 0
        assert torch.equal(_bits(kc), _bits(kr)) and torch.equal(_bits(vc), _bits(vr))
        flat = kc.cpu().reshape(-1, Hkv, d)
        for b, slot in enumerate(slots):
            assert torch.equal(_bits(flat[slot]), _bits(key[b]))
        assert _max_err(out, ref) <= ATOL_16
