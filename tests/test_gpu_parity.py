"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: slot mapping, store and unpack bit-exact; attention max abs error
<= 2e-2 for fp16/bf16 caches and <= 1e-5 for fp32 caches against the
binary64 oracle.  Small cases span several pipeline stages and partitions
and end in ragged tails (NaN-filled, so any masked-row leak shows); the
full-size cases run the workloads in the benchmark's launch configuration.
"""
import pytest
import torch

import pkv_workloads as wl
from conftest import attn_error, load_golden

pytestmark = pytest.mark.gpu

ATOL_16 = 2e-2
ATOL_32 = 1e-5


def _zero_err(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def _max_err(out, ref):
    return attn_error(out, ref)


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


# ------------------------------------------------------------------ page-3 walk
def test_tiny_walk_trace(pkv, orc, cuda_dev):
    golden = load_golden("walk_trace.json")["derived_by_the_page_rules"]["steps"]
    tr = wl.tiny_trace(seed=0, device=cuda_dev)
    err = _zero_err(cuda_dev)
    kc, vc = tr.k_cache0.clone(), tr.v_cache0.clone()
    kc_ref, vc_ref = tr.k_cache0.cpu(), tr.v_cache0.cpu()
    for st, gold in zip(tr.steps, golden):
        n = int(st["cu_new"][-1])
        slots = pkv.pkv_compute_slot_mapping(st["block_tables"], st["starts"], st["ends"], st["cu_new"], 4, 8,
                                             num_new_tokens=n, err_flag=err)
        want, _ = orc.compute_slot_mapping(st["block_tables"], st["starts"], st["ends"], 4, 8)
        assert slots.cpu().tolist() == want.tolist() == gold["slots"]
        pkv.pkv_store_kvcache(st["key"], st["value"], kc, vc, slots, err_flag=err)
        kc_ref, vc_ref, _ = orc.store_kvcache(st["key"], st["value"], kc_ref, vc_ref, want)
        assert torch.equal(_bits(kc), _bits(kc_ref)) and torch.equal(_bits(vc), _bits(vc_ref))
        out = pkv.pkv_paged_attention_decode(st["q"], kc, vc, st["block_tables"], st["context_lens"], 0.5, 8,
                                             err_flag=err)
        ref, _ = orc.paged_attention_decode(st["q"], kc_ref, vc_ref, st["block_tables"], st["context_lens"], 0.5)
        assert _max_err(out, ref) <= ATOL_32
    assert int(err.item()) == 0


# ------------------------------------------------------------------ slot mapping
@pytest.mark.parametrize("bs", [4, 16, 256])
def test_slot_mapping_ranges(pkv, orc, cuda_dev, bs):
    g = torch.Generator().manual_seed(bs)
    B, nb = 13, 64
    lens = torch.randint(0, 5 * bs, (B,), generator=g)
    perm = torch.randperm(nb, generator=g).tolist()
    maxb = max(1, max((int(x) + bs - 1) // bs for x in lens))
    bt = torch.full((B, maxb), -1, dtype=torch.int32)
    k = 0
    for b in range(B):
        m = (int(lens[b]) + bs - 1) // bs
        bt[b, :m] = torch.tensor(perm[k:k + m], dtype=torch.int32) if m else bt[b, :0]
        k += m
    starts = torch.stack([torch.randint(0, int(n) + 1, (1,), generator=g)[0] for n in lens]).to(torch.int32)
    ends = torch.stack([torch.randint(int(s), int(n) + 1, (1,), generator=g)[0]
                        for s, n in zip(starts, lens)]).to(torch.int32)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(ends - starts, 0)
    err = _zero_err(cuda_dev)
    got = pkv.pkv_compute_slot_mapping(bt.to(cuda_dev), starts.to(cuda_dev), ends.to(cuda_dev), cu.to(cuda_dev),
                                       bs, nb, num_new_tokens=int(cu[-1]), err_flag=err)
    want, nerr = orc.compute_slot_mapping(bt, starts, ends, bs, nb)
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(got.cpu(), want)


def test_slot_mapping_errors(pkv, orc, cuda_dev):
    bt = torch.tensor([[7, -1], [9, 1]], dtype=torch.int32)  # -1 inside the range; 9 >= num_blocks
    starts, ends = torch.tensor([2, 0], dtype=torch.int32), torch.tensor([6, 5], dtype=torch.int32)
    cu = torch.tensor([0, 4, 9], dtype=torch.int32)
    err = _zero_err(cuda_dev)
    got = pkv.pkv_compute_slot_mapping(bt.to(cuda_dev), starts.to(cuda_dev), ends.to(cuda_dev), cu.to(cuda_dev),
                                       4, 8, num_new_tokens=9, err_flag=err)
    want, nerr = orc.compute_slot_mapping(bt, starts, ends, 4, 8)
    assert torch.equal(got.cpu(), want) and nerr == 6
    assert int(err.item()) & pkv.ERRBIT_BLOCK_RANGE
    # a span that disagrees with [start, end) is flagged and never overruns the output
    err.zero_()
    bad_cu = torch.tensor([0, 3, 9], dtype=torch.int32)
    out = torch.full((9,), -7, dtype=torch.int32, device=cuda_dev)
    pkv.pkv_compute_slot_mapping(bt.to(cuda_dev), starts.to(cuda_dev), ends.to(cuda_dev), bad_cu.to(cuda_dev), 4,
                                 8, out=out, err_flag=err)
    assert int(err.item()) & pkv.ERRBIT_SPAN


# ------------------------------------------------------------------ store_kvcache
@pytest.mark.parametrize("dtype,H,d,bs", [(torch.float32, 2, 4, 4), (torch.bfloat16, 8, 128, 16),
                                          (torch.float16, 32, 128, 16), (torch.float16, 3, 5, 8),
                                          (torch.bfloat16, 1, 8, 256)])
def test_store_parity(pkv, orc, cuda_dev, dtype, H, d, bs):
    g = torch.Generator().manual_seed(H * 1000 + d)
    N = 150
    nb = max(24, (2 * N + bs - 1) // bs)
    kc = torch.randn(nb, bs, H, d, generator=g).to(dtype)
    vc = torch.randn(nb, bs, H, d, generator=g).to(dtype)
    key = torch.randn(N, H, d, generator=g).to(dtype)
    value = torch.randn(N, H, d, generator=g).to(dtype)
    slots = torch.randperm(nb * bs, generator=g)[:N].to(torch.int32)
    slots[::7] = -1
    err = _zero_err(cuda_dev)
    kd, vd = kc.to(cuda_dev), vc.to(cuda_dev)
    pkv.pkv_store_kvcache(key.to(cuda_dev), value.to(cuda_dev), kd, vd, slots.to(cuda_dev), err_flag=err)
    kr, vr, nerr = orc.store_kvcache(key, value, kc, vc, slots)
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(_bits(kd), _bits(kr)) and torch.equal(_bits(vd), _bits(vr))


def test_store_bad_slots_are_skipped(pkv, orc, cuda_dev):
    nb, bs, H, d = 4, 16, 2, 64
    kc = torch.zeros(nb, bs, H, d, dtype=torch.bfloat16)
    key = torch.ones(4, H, d, dtype=torch.bfloat16)
    slots = torch.tensor([3, nb * bs, -5, 10], dtype=torch.int32)
    err = _zero_err(cuda_dev)
    kd, vd = kc.to(cuda_dev), kc.clone().to(cuda_dev)
    pkv.pkv_store_kvcache(key.to(cuda_dev), key.to(cuda_dev), kd, vd, slots.to(cuda_dev), err_flag=err)
    kr, _, nerr = orc.store_kvcache(key, key, kc, kc.clone(), slots)
    assert nerr == 2 and int(err.item()) == pkv.ERRBIT_SLOT_RANGE
    assert torch.equal(_bits(kd), _bits(kr))


# ------------------------------------------------------------------ attention: tensor-core path
FAST_HEADS = [(8, 8), (16, 8), (32, 8), (8, 1), (4, 2), (16, 2), (64, 8)]  # G = 1, 2, 4, 8, 2, 8, 8


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", FAST_HEADS)
@pytest.mark.parametrize("bs", [16, 32, 256])
def test_decode_fast_path(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs):
    lens = [0, 1, 15, 16, 17, 100, 1000, 2100]
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, len(lens), 1, 2100, 400)
    batch = wl.decode_batch(cfg, seed=Hq * 7 + Hkv + bs, device=cuda_dev, ctx_override=lens, nan_tails=True,
                            nan_unused=True)
    part, nparts, fast = pkv.pkv_paged_attention_decode_plan(len(lens), Hq, Hkv, 128, bs, 2100, dtype)
    assert fast and part == 0 and nparts >= 1
    err = _zero_err(cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, 2100, err_flag=err)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[0]) == 0  # context length 0 -> zero row


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_single_token_is_exact_v_row(pkv, cuda_dev, dtype):
    cfg = wl.DecodeConfig("t", dtype, 32, 8, 128, 16, 3, 1, 1, 40)
    batch = wl.decode_batch(cfg, seed=5, device=cuda_dev, ctx_override=[1, 1, 1], q_gain=8.0)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, 1)
    for b in range(3):
        blk = int(batch.block_tables[b, 0])
        want = batch.v_cache[blk, 0].repeat_interleave(4, 0)  # [Hq, d]
        assert torch.equal(_bits(out[b]), _bits(want))


def test_decode_peaky_softmax_and_split_invariance(pkv, orc, cuda_dev):
    """A sequence's result does not depend on how the work-balanced schedule cuts
    it: alone it is spread over every CTA, inside a batch over a few, and with
    more than 1024 sequences the fixed-partition kernel takes it."""
    cfg = wl.LONG_GQA_8K
    lens = [5000, 777, 4096, 1]
    batch = wl.decode_batch(cfg, seed=9, device=cuda_dev, batch=4, ctx_override=lens, q_gain=8.0, nan_tails=True)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    full = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                          batch.context_lens, batch.scale, 5000)
    assert _max_err(full, ref) <= ATOL_16
    for b in range(4):  # each sequence alone
        one = pkv.pkv_paged_attention_decode(batch.q[b:b + 1].contiguous(), batch.k_cache, batch.v_cache,
                                             batch.block_tables[b:b + 1].contiguous(),
                                             batch.context_lens[b:b + 1].contiguous(), batch.scale, 5000)
        assert _max_err(one[0], ref[b]) <= ATOL_16
        assert (one[0].float() - full[b].float()).abs().max().item() <= 1e-2


EQUAL_CASES = [(32, 8, 16, 3000, 3), (16, 8, 16, 300, 5), (8, 8, 256, 40, 3), (4, 1, 16, 1, 7),
               (64, 8, 32, 1000, 2), (8, 2, 16, 17, 40), (16, 8, 16, 700, 100)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv,bs,ctx,B", EQUAL_CASES)
def test_decode_equal_lengths(pkv, orc, cuda_dev, dtype, Hq, Hkv, bs, ctx, B):
    """Every sequence at max_ctx: the schedule the producer guesses from
    max_ctx is the real one, and its first stages' copies leave before the
    plan is computed.  Short units (no tail), one-token contexts, units split
    over many CTAs and batches of up to 128 sequences all match the oracle."""
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, 128, bs, B, 1, ctx, None)
    batch = wl.decode_batch(cfg, seed=ctx + B, device=cuda_dev, ctx_override=[ctx] * B, nan_tails=True,
                            nan_unused=True)
    err = _zero_err(cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, ctx, err_flag=err)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16


@pytest.mark.parametrize("B,Hq,Hkv", [(64, 16, 8), (40, 32, 8), (200, 32, 8), (512, 64, 8)])
def test_decode_merge_row_layouts(pkv, orc, cuda_dev, B, Hq, Hkv):
    """The piece merge shares a row among 8, 4, 2 or 1 warps depending on how
    many (unit, query head) rows a launch has (1024, 1280, 6400 and 32768
    rows here); every layout matches the oracle on split units."""
    g = torch.Generator().manual_seed(B + Hq)
    hi = 3000 if B < 100 else 600  # keeps the oracle's work to a few seconds
    lens = torch.randint(1, hi, (B,), generator=g)
    lens[:3] = torch.tensor([0, hi - 1, 1])
    cfg = wl.DecodeConfig("t", torch.bfloat16, Hq, Hkv, 128, 16, B, 1, hi, None)
    batch = wl.decode_batch(cfg, seed=B, device=cuda_dev, ctx_override=lens.tolist(), nan_tails=True)
    err = _zero_err(cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, hi, err_flag=err)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16
    assert torch.count_nonzero(out[0]) == 0


def test_decode_fixed_partition_kernel_for_large_batches(pkv, orc, cuda_dev):
    """More than 512 sequences of a 16-bit cache use the tensor-core kernel
    with fixed partitions of the context (and the split-K combine for the long
    ones)."""
    g = torch.Generator().manual_seed(77)
    B = 1100
    lens = torch.randint(1, 200, (B,), generator=g)
    lens[:5] = torch.tensor([3000, 1234, 16, 17, 0])
    cfg = wl.DecodeConfig("t", torch.bfloat16, 8, 4, 128, 16, B, 1, 3000, 20000)
    batch = wl.decode_batch(cfg, seed=78, device=cuda_dev, ctx_override=lens.tolist(), nan_tails=True)
    part, nparts, fast = pkv.pkv_paged_attention_decode_plan(B, 8, 4, 128, 16, 3000, torch.bfloat16)
    assert fast and part > 0 and nparts > 1
    err = _zero_err(cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, 3000, err_flag=err)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    assert int(err.item()) == 0
    assert _max_err(out, ref) <= ATOL_16


def test_decode_unaligned_pools_fall_back_within_the_workspace(pkv, orc, cuda_dev):
    """Pools that are not 16-byte aligned cannot feed TMA: the call runs the
    CUDA-core kernel with partitions that fit the size-query workspace."""
    cfg = wl.DecodeConfig("t", torch.bfloat16, 16, 8, 128, 16, 3, 1, 3000, 500)
    batch = wl.decode_batch(cfg, seed=79, device=cuda_dev, ctx_override=[3000, 1, 999])
    flat_k = torch.empty(batch.k_cache.numel() + 1, dtype=cfg.dtype, device=cuda_dev)
    flat_v = torch.empty_like(flat_k)
    kc = flat_k[1:].view(batch.k_cache.shape)
    vc = flat_v[1:].view(batch.v_cache.shape)
    kc.copy_(batch.k_cache)
    vc.copy_(batch.v_cache)
    assert kc.data_ptr() % 16 != 0
    out = pkv.pkv_paged_attention_decode(batch.q, kc, vc, batch.block_tables, batch.context_lens, batch.scale, 3000)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    assert _max_err(out, ref) <= ATOL_16


def test_decode_error_semantics(pkv, orc, cuda_dev):
    cfg = wl.DecodeConfig("t", torch.bfloat16, 16, 8, 128, 16, 4, 1, 600, 200)
    batch = wl.decode_batch(cfg, seed=13, device=cuda_dev, ctx_override=[300, 600, 0, 50])
    bt = batch.block_tables.clone()
    bt[0, 3] = 10_000          # used block id out of range: its 16 tokens are dropped
    err = _zero_err(cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, bt, batch.context_lens,
                                         batch.scale, 600, err_flag=err)
    ref, nerr = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, bt, batch.context_lens,
                                           batch.scale)
    assert nerr == 1 and int(err.item()) == pkv.ERRBIT_BLOCK_RANGE
    assert _max_err(out, ref) <= ATOL_16
    # a context longer than the declared bound: zero row and PKV_ERRBIT_CONTEXT
    err.zero_()
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, 400, err_flag=err)
    assert int(err.item()) & pkv.ERRBIT_CONTEXT
    assert torch.count_nonzero(out[1]) == 0
    ref2, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale)
    keep = [0, 2, 3]
    assert _max_err(out[keep], ref2[keep]) <= ATOL_16


# ------------------------------------------------------------------ attention: CUDA-core path
@pytest.mark.parametrize("bs", [4, 16, 256])
def test_decode_generic_fp32_page_case(pkv, orc, cuda_dev, bs):
    """The page's Step 2 shapes: Hq 4, Hkv 2, d 8, lens [1, bs, 2bs+3], fp32."""
    lens = [1, bs, 2 * bs + 3]
    cfg = wl.DecodeConfig("t", torch.float32, 4, 2, 8, bs, 3, 1, 2 * bs + 3, 12)
    batch = wl.decode_batch(cfg, seed=bs, device=cuda_dev, ctx_override=lens, nan_tails=True)
    scale = 8 ** -0.5
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, scale, 2 * bs + 3)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, scale)
    assert _max_err(out, ref) <= ATOL_32


@pytest.mark.parametrize("dtype,Hq,Hkv,d,bs,tol", [
    (torch.float32, 8, 2, 128, 16, ATOL_32),    # fp32, long: several partitions + combine
    (torch.float16, 8, 4, 64, 16, ATOL_16),     # head_dim 64
    (torch.bfloat16, 32, 2, 128, 16, ATOL_16),  # G = 16 > 8
    (torch.bfloat16, 4, 4, 128, 8, ATOL_16),    # block size not a multiple of 16
])
def test_decode_generic_path(pkv, orc, cuda_dev, dtype, Hq, Hkv, d, bs, tol):
    lens = [3, 300, 1500, 0, 2222]
    cfg = wl.DecodeConfig("t", dtype, Hq, Hkv, d, bs, len(lens), 1, 2222, None)
    batch = wl.decode_batch(cfg, seed=d + Hq, device=cuda_dev, ctx_override=lens, nan_tails=True)
    assert not pkv.pkv_paged_attention_decode_plan(len(lens), Hq, Hkv, d, bs, 2222, dtype)[2]
    err = _zero_err(cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, 2222, err_flag=err)
    ref, _ = orc.paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                        batch.context_lens, batch.scale)
    assert int(err.item()) == 0
    assert _max_err(out, ref) <= tol


# ------------------------------------------------------------------ unpack
@pytest.mark.parametrize("dtype,H,d,idx", [(torch.bfloat16, 8, 128, torch.int32), (torch.bfloat16, 8, 128, torch.int64),
                                           (torch.float32, 2, 8, torch.int32), (torch.float16, 3, 5, torch.int64)])
def test_unpack_parity(pkv, orc, cuda_dev, dtype, H, d, idx):
    cfg = wl.CsrConfig("t", dtype, 16, H, d, 40, 96, 0.5, 1, 300, idx)
    snap = wl.csr_snapshot(cfg, seed=H + d, device=cuda_dev)
    pkv.pkv_validate_index_buffers(snap.seq_ptr.cpu(), snap.block_table.cpu(), snap.unique_pages)
    pkv.pkv_validate_token_ptr(snap.token_ptr.cpu(), snap.seq_ptr.cpu(), 16, snap.total_tokens)
    err = _zero_err(cuda_dev)
    got = pkv.pkv_unpack_block_paged(snap.k_pool, snap.block_table, snap.seq_ptr, snap.token_ptr,
                                     total_tokens=snap.total_tokens, err_flag=err)
    want, nerr = orc.unpack_block_paged(snap.k_pool, snap.block_table, snap.seq_ptr, snap.token_ptr, index_dtype=idx)
    assert nerr == 0 and int(err.item()) == 0
    assert torch.equal(_bits(got), _bits(want))
    # aliased prefix: every sharing sequence's first 96 rows are the same bytes
    tp = snap.token_ptr.cpu()
    for s in range(1, 20):
        assert torch.equal(_bits(got[tp[s]:tp[s] + 96]), _bits(got[0:96]))


def test_unpack_errors_zero_fill(pkv, orc, cuda_dev):
    pool = torch.randn(6, 4, 2, 8).to(torch.bfloat16)
    bt = torch.tensor([0, 9, 2, 3], dtype=torch.int32)     # page id 9 >= num_pages
    sp = torch.tensor([0, 2, 3, 4], dtype=torch.int32)
    tp = torch.tensor([0, 8, 14, 16], dtype=torch.int64)   # seq 1 needs 2 pages, owns 1
    err = _zero_err(cuda_dev)
    got = pkv.pkv_unpack_block_paged(pool.to(cuda_dev), bt.to(cuda_dev), sp.to(cuda_dev), tp.to(cuda_dev),
                                     total_tokens=16, err_flag=err)
    want, nerr = orc.unpack_block_paged(pool, bt, sp, tp, index_dtype=torch.int32)
    assert nerr > 0
    assert int(err.item()) == pkv.ERRBIT_CSR_PHYS | pkv.ERRBIT_CSR_PAGE
    assert torch.equal(_bits(got), _bits(want))


# ------------------------------------------------------------------ full-size workloads
DECODE_CONFIGS = ["llama2-7b-layer-fp16", "qwen3-0.6b-gqa-bf16", "long-gqa-8k-bf16", "long-gqa-32k-bf16"]


@pytest.mark.parametrize("name", DECODE_CONFIGS)
def test_full_size_decode_step(pkv, orc, cuda_dev, name):
    """One decode step at the workload's full size: slot mapping and store of
    the new token (bit-exact over the whole caches), then attention over every
    sequence and head against the oracle."""
    cfg = wl.CONFIGS[name]
    batch = wl.decode_batch(cfg, seed=1, device=cuda_dev, nan_tails=True)
    B, bs, nb = cfg.batch, cfg.block_size, batch.extra["num_blocks"]
    err = _zero_err(cuda_dev)
    kc0, vc0 = batch.k_cache.cpu(), batch.v_cache.cpu()
    slots = pkv.pkv_compute_slot_mapping(batch.block_tables, batch.starts, batch.ends, batch.cu_new, bs, nb,
                                         num_new_tokens=B, err_flag=err)
    want_slots, _ = orc.compute_slot_mapping(batch.block_tables, batch.starts, batch.ends, bs, nb)
    assert torch.equal(slots.cpu(), want_slots)
    pkv.pkv_store_kvcache(batch.new_key, batch.new_value, batch.k_cache, batch.v_cache, slots, err_flag=err)
    kr, vr, _ = orc.store_kvcache(batch.new_key, batch.new_value, kc0, vc0, want_slots)
    del kc0, vc0
    assert torch.equal(_bits(batch.k_cache), _bits(kr)) and torch.equal(_bits(batch.v_cache), _bits(vr))
    ws = pkv.pkv_paged_attention_decode_workspace_size(B, cfg.num_q_heads, cfg.num_kv_heads, 128, bs,
                                                       batch.max_context_len, cfg.dtype)
    workspace = torch.zeros(max(ws, 1), dtype=torch.uint8, device=cuda_dev)
    out = pkv.pkv_paged_attention_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                         batch.context_lens, batch.scale, batch.max_context_len,
                                         workspace=workspace, err_flag=err)
    ref, _ = orc.paged_attention_decode(batch.q, kr, vr, batch.block_tables, batch.context_lens, batch.scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not torch.isnan(out).any()
    assert _max_err(out, ref) <= ATOL_16


def test_full_size_csr_snapshot(pkv, orc, cuda_dev):
    """The prefix-shared snapshot: unpack of both roles bit-exact, and decode
    attention over the same pages (Hq == Hkv == num_heads)."""
    snap = wl.csr_snapshot(wl.CSR_PREFIX, seed=2, device=cuda_dev)
    err = _zero_err(cuda_dev)
    for pool in (snap.k_pool, snap.v_pool):
        got = pkv.pkv_unpack_block_paged(pool, snap.block_table, snap.seq_ptr, snap.token_ptr,
                                         total_tokens=snap.total_tokens, err_flag=err)
        want, nerr = orc.unpack_block_paged(pool, snap.block_table, snap.seq_ptr, snap.token_ptr,
                                            index_dtype=snap.block_table.dtype)
        assert nerr == 0
        assert torch.equal(_bits(got), _bits(want))
        del got, want
    maxc = int(snap.seq_lens.max())
    out = pkv.pkv_paged_attention_decode(snap.q, snap.k_pool, snap.v_pool, snap.block_tables_2d, snap.seq_lens,
                                         snap.scale, maxc, err_flag=err)
    ref, _ = orc.paged_attention_decode(snap.q, snap.k_pool, snap.v_pool, snap.block_tables_2d, snap.seq_lens,
                                        snap.scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _max_err(out, ref) <= ATOL_16
