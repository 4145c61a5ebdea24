"""Seeded synthetic inputs for the paged-KV hot path.

This module builds inputs only: random tensors, random block assignments,
context lengths and the CSR index buffers of a snapshot.  It holds none of the
method's arithmetic (no slot formula, no gather, no attention), so the CUDA
path and the CPU oracle can both be fed from it without sharing any code.

The workload shapes follow the pages' worked examples and model arithmetic:
  * the four-token-block example of "Paged KV Cache - AI infra interview
    lesson" ("Walk the Shapes First");
  * a LLaMA-2-7B-shaped layer and a Qwen3-0.6B-shaped GQA layer (same page,
    "Why It Matters");
  * long-context GQA sequences of 8192 and 32768 tokens (the "Illustrative
    arithmetic" of "Chapter 2 - KV cache, memory hierarchy, continuous batching,
    and PagedAttention" scaled to one layer);
  * a CSR block-paged snapshot with aliased prefix pages ("Block-Paged KV
    Cache", "Element lookup through the block table").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    batch: int
    ctx_lo: int
    ctx_hi: int
    num_blocks: int | None  # None: exactly the blocks the batch needs
    description: str = ""


@dataclass(frozen=True)
class CsrConfig:
    name: str
    dtype: torch.dtype
    page_size: int
    num_heads: int
    head_dim: int
    num_seqs: int
    prefix_tokens: int
    shared_fraction: float
    suffix_lo: int
    suffix_hi: int
    index_dtype: torch.dtype = torch.int32  # u32 index buffers (values < 2^31)
    description: str = ""


@dataclass(frozen=True)
class TinyConfig:
    name: str = "tiny-walk-fp32"
    dtype: torch.dtype = torch.float32
    block_size: int = 4
    num_kv_heads: int = 2
    num_q_heads: int = 4
    head_dim: int = 4
    num_blocks: int = 8
    description: str = ("page-3 walk: block_size 4, Hkv 2, Hq 4, d 4, 8 blocks; seq A 6 tokens "
                        "table [7,2], seq B 3 tokens table [5]; prefill + 2 decode steps")


TINY = TinyConfig()
LLAMA2_7B_LAYER = DecodeConfig(
    "llama2-7b-layer-fp16", torch.float16, 32, 32, 128, 16, 64, 1, 4096, 20000,
    "LLaMA-2-7B-shaped layer: Hq=Hkv=32, d=128, bs=16, B=64, ctx~U[1,4096], 20000-block pool")
QWEN3_GQA = DecodeConfig(
    "qwen3-0.6b-gqa-bf16", torch.bfloat16, 16, 8, 128, 256, 128, 256, 8192, 4096,
    "Qwen3-0.6B-shaped GQA layer: Hq=16, Hkv=8, d=128, bs=256, B=128, ctx~U[256,8192]")
QWEN3_GQA_B1024 = DecodeConfig(
    "qwen3-0.6b-gqa-bf16-b1024", torch.bfloat16, 16, 8, 128, 256, 1024, 256, 8192, None,
    "Qwen3-0.6B-shaped GQA layer at a serving batch of 1024 sequences: Hq=16, Hkv=8, d=128, bs=256, "
    "ctx~U[256,8192], pool of exactly the blocks the batch needs")
LONG_GQA_8K = DecodeConfig(
    "long-gqa-8k-bf16", torch.bfloat16, 32, 8, 128, 16, 8, 8192, 8192, None,
    "long-context GQA: Hq=32, Hkv=8, d=128, bs=16, 8 sequences x 8192 tokens")
LONG_GQA_32K = DecodeConfig(
    "long-gqa-32k-bf16", torch.bfloat16, 32, 8, 128, 16, 8, 32768, 32768, None,
    "long-context GQA: Hq=32, Hkv=8, d=128, bs=16, 8 sequences x 32768 tokens")
CSR_PREFIX = CsrConfig(
    "csr-prefix-bf16", torch.bfloat16, 16, 8, 128, 256, 1024, 0.5, 1, 2048, torch.int32,
    "CSR snapshot: page_size=16, H=8, d=128, 256 seqs, half share a 1024-token aliased prefix, "
    "suffix~U[1,2048], u32 index buffers")

CONFIGS = {c.name: c for c in (TINY, LLAMA2_7B_LAYER, QWEN3_GQA, QWEN3_GQA_B1024, LONG_GQA_8K, LONG_GQA_32K,
                                CSR_PREFIX)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, dtype, device, gen):
    if dtype == torch.float32:
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    # draw in fp32 then round once, so every storage type sees N(0,1) samples
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


@dataclass
class DecodeBatch:
    cfg: DecodeConfig
    q: torch.Tensor               # [B, Hq, d]
    k_cache: torch.Tensor         # [num_blocks, bs, Hkv, d]
    v_cache: torch.Tensor
    block_tables: torch.Tensor    # int32 [B, max_blocks], -1 padded
    context_lens: torch.Tensor    # int32 [B], includes the token written this step
    new_key: torch.Tensor         # [B, Hkv, d]: K/V of the token at position ctx-1
    new_value: torch.Tensor
    starts: torch.Tensor          # int32 [B]: first position written this step (ctx-1)
    ends: torch.Tensor            # int32 [B]: one past the last (ctx)
    cu_new: torch.Tensor          # int32 [B+1]: offsets of each sequence's new tokens
    scale: float
    max_context_len: int
    extra: dict = field(default_factory=dict)

    @property
    def kv_bytes(self) -> int:
        """KV bytes one decode step reads: sum_b ctx_b * 2 * Hkv * d * elem (M_KV with L=1)."""
        c = self.cfg
        es = torch.tensor([], dtype=c.dtype).element_size()
        return int(self.context_lens.to(torch.int64).sum()) * 2 * c.num_kv_heads * c.head_dim * es


def decode_batch(cfg: DecodeConfig, seed: int = 0, device="cpu", *, nan_tails=False,
                 nan_unused=False, batch: int | None = None, ctx_override=None,
                 q_gain: float = 1.0) -> DecodeBatch:
    """One decode step's inputs for a decode config.

    Context lengths ~ U[ctx_lo, ctx_hi]; each sequence's blocks are a random,
    non-contiguous draw from the pool (a prefix of one random permutation).
    nan_tails fills the unused rows of every last block with NaN, nan_unused
    fills every block no table references with NaN: any read of a masked or
    unreferenced row then shows up in the output.  q_gain scales q (a value
    of 8 gives a peaky softmax).
    """
    if batch is not None or ctx_override is not None:
        cfg = replace(cfg, batch=batch if batch is not None else cfg.batch)
    gc = _gen(seed, "cpu")
    B, bs = cfg.batch, cfg.block_size
    if ctx_override is not None:
        ctx = torch.as_tensor(ctx_override, dtype=torch.int32).reshape(B)
    else:
        ctx = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (B,), generator=gc, dtype=torch.int64)
        ctx = ctx.to(torch.int32)
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    need = sum(nblk)
    num_blocks = cfg.num_blocks if cfg.num_blocks is not None else max(need, 1)
    if need > num_blocks:
        raise ValueError(f"{cfg.name}: batch needs {need} blocks, pool has {num_blocks}")
    perm = torch.randperm(num_blocks, generator=gc)[:need].tolist()
    max_blocks = max([(cfg.ctx_hi + bs - 1) // bs] + nblk + [1])
    tables = torch.full((B, max_blocks), -1, dtype=torch.int32)
    k = 0
    for b in range(B):
        tables[b, : nblk[b]] = torch.tensor(perm[k: k + nblk[b]], dtype=torch.int32)
        k += nblk[b]

    gd = _gen(seed + 1000, device)
    shape = (num_blocks, bs, cfg.num_kv_heads, cfg.head_dim)
    k_cache = _randn(shape, cfg.dtype, device, gd)
    v_cache = _randn(shape, cfg.dtype, device, gd)
    q = _randn((B, cfg.num_q_heads, cfg.head_dim), cfg.dtype, device, gd)
    if q_gain != 1.0:
        q = (q.float() * q_gain).to(cfg.dtype)
    new_key = _randn((B, cfg.num_kv_heads, cfg.head_dim), cfg.dtype, device, gd)
    new_value = _randn((B, cfg.num_kv_heads, cfg.head_dim), cfg.dtype, device, gd)

    if nan_unused:
        used = torch.zeros(num_blocks, dtype=torch.bool)
        used[torch.tensor(perm[:need], dtype=torch.int64)] = True
        unused = (~used).nonzero().flatten().to(device)
        k_cache[unused] = float("nan")
        v_cache[unused] = float("nan")
    if nan_tails:
        for b in range(B):
            n = int(ctx[b])
            if n == 0:
                continue
            filled = n - (nblk[b] - 1) * bs
            if filled < bs:
                last = int(tables[b, nblk[b] - 1])
                k_cache[last, filled:] = float("nan")
                v_cache[last, filled:] = float("nan")

    starts = (ctx - 1).clamp(min=0).to(torch.int32)
    ends = ctx.clone()
    cu_new = torch.zeros(B + 1, dtype=torch.int32)
    cu_new[1:] = torch.cumsum(ends - starts, 0).to(torch.int32)
    return DecodeBatch(cfg=cfg, q=q, k_cache=k_cache, v_cache=v_cache,
                       block_tables=tables.to(device), context_lens=ctx.to(device),
                       new_key=new_key, new_value=new_value, starts=starts.to(device),
                       ends=ends.to(device), cu_new=cu_new.to(device),
                       scale=1.0 / math.sqrt(cfg.head_dim),
                       max_context_len=max(int(ctx.max()) if B else 0, 0),
                       extra={"num_blocks": num_blocks})


@dataclass
class CsrSnapshot:
    cfg: CsrConfig
    k_pool: torch.Tensor       # [num_pages, page_size, H, d]
    v_pool: torch.Tensor
    block_table: torch.Tensor  # [nnz] (index dtype)
    seq_ptr: torch.Tensor      # [S+1] (index dtype)
    token_ptr: torch.Tensor    # int64 [S+1]: sequence s owns logical rows token_ptr[s]..[s+1]-1
    seq_lens: torch.Tensor     # int32 [S]
    block_tables_2d: torch.Tensor  # int32 [S, max_pages], -1 padded (same pages, for attention)
    q: torch.Tensor            # [S, H, d] for attention over the snapshot (Hq == Hkv == H)
    scale: float
    unique_pages: int

    @property
    def total_tokens(self) -> int:
        return int(self.token_ptr[-1])


def csr_snapshot(cfg: CsrConfig = CSR_PREFIX, seed: int = 0, device="cpu", *,
                 num_seqs: int | None = None, prefix_tokens: int | None = None,
                 suffix_hi: int | None = None) -> CsrSnapshot:
    """A block-paged snapshot in which the first shared_fraction of the sequences
    name the same prefix pages (aliasing), followed by private suffix pages."""
    if num_seqs is not None or prefix_tokens is not None or suffix_hi is not None:
        cfg = replace(cfg, num_seqs=num_seqs or cfg.num_seqs,
                      prefix_tokens=cfg.prefix_tokens if prefix_tokens is None else prefix_tokens,
                      suffix_hi=suffix_hi or cfg.suffix_hi)
    gc = _gen(seed, "cpu")
    S, ps = cfg.num_seqs, cfg.page_size
    assert cfg.prefix_tokens % ps == 0, "the shared prefix is page-aligned"
    n_prefix_pages = cfg.prefix_tokens // ps
    n_shared = int(S * cfg.shared_fraction)
    suffix = torch.randint(cfg.suffix_lo, cfg.suffix_hi + 1, (S,), generator=gc, dtype=torch.int64)
    suffix_pages = [(int(x) + ps - 1) // ps for x in suffix]
    total_pages = n_prefix_pages + sum(suffix_pages)
    perm = torch.randperm(total_pages, generator=gc).tolist()
    prefix_ids = perm[:n_prefix_pages]
    k = n_prefix_pages
    pages, lens = [], []
    for s in range(S):
        own = perm[k: k + suffix_pages[s]]
        k += suffix_pages[s]
        if s < n_shared:
            pages.append(prefix_ids + own)
            lens.append(cfg.prefix_tokens + int(suffix[s]))
        else:
            pages.append(own)
            lens.append(int(suffix[s]))
    counts = torch.tensor([len(p) for p in pages], dtype=torch.int64)
    seq_ptr = torch.zeros(S + 1, dtype=torch.int64)
    seq_ptr[1:] = torch.cumsum(counts, 0)
    block_table = torch.tensor([x for p in pages for x in p], dtype=torch.int64)
    seq_lens = torch.tensor(lens, dtype=torch.int64)
    token_ptr = torch.zeros(S + 1, dtype=torch.int64)
    token_ptr[1:] = torch.cumsum(seq_lens, 0)
    max_pages = int(counts.max()) if S else 1
    bt2d = torch.full((S, max_pages), -1, dtype=torch.int32)
    for s in range(S):
        bt2d[s, : len(pages[s])] = torch.tensor(pages[s], dtype=torch.int32)

    gd = _gen(seed + 1000, device)
    shape = (total_pages, ps, cfg.num_heads, cfg.head_dim)
    k_pool = _randn(shape, cfg.dtype, device, gd)
    v_pool = _randn(shape, cfg.dtype, device, gd)
    q = _randn((S, cfg.num_heads, cfg.head_dim), cfg.dtype, device, gd)
    idt = cfg.index_dtype
    return CsrSnapshot(cfg=cfg, k_pool=k_pool, v_pool=v_pool,
                       block_table=block_table.to(idt).to(device),
                       seq_ptr=seq_ptr.to(idt).to(device), token_ptr=token_ptr.to(device),
                       seq_lens=seq_lens.to(torch.int32).to(device),
                       block_tables_2d=bt2d.to(device), q=q, scale=1.0 / math.sqrt(cfg.head_dim),
                       unique_pages=total_pages)


@dataclass
class TinyTrace:
    """Page-3 walk: one prefill then two decode steps for sequences A and B.

    Reading of the walk (the page's table did not survive extraction; its
    rules did): A holds 6 tokens in blocks [7, 2], B holds 3 tokens in block
    [5]; each decode step adds one token per sequence; B's fifth token
    (len 5, 5 % 4 == 1) needs a new block, taken as the lowest-numbered free
    block (0).  Each step lists the block tables after allocation, the
    positions written ([start, end) per sequence) and the context lengths.
    """
    cfg: TinyConfig
    steps: list          # list of dicts: block_tables, starts, ends, context_lens, key, value, q
    k_cache0: torch.Tensor
    v_cache0: torch.Tensor


def tiny_trace(seed: int = 0, device="cpu") -> TinyTrace:
    cfg = TINY
    g = _gen(seed, "cpu")
    H, d, Hq, bs = cfg.num_kv_heads, cfg.head_dim, cfg.num_q_heads, cfg.block_size
    tables = [
        [[7, 2, -1], [5, -1, -1]],   # prefill
        [[7, 2, -1], [5, -1, -1]],   # decode 1: A len 7, B len 4
        [[7, 2, -1], [5, 0, -1]],    # decode 2: A len 8, B len 5 -> new block 0
    ]
    spans = [([0, 0], [6, 3]), ([6, 3], [7, 4]), ([7, 4], [8, 5])]
    steps = []
    for bt, (st, en) in zip(tables, spans):
        n = sum(e - s for s, e in zip(st, en))
        cu = [0, en[0] - st[0], en[0] - st[0] + en[1] - st[1]]
        steps.append(dict(
            cu_new=torch.tensor(cu, dtype=torch.int32).to(device),
            block_tables=torch.tensor(bt, dtype=torch.int32).to(device),
            starts=torch.tensor(st, dtype=torch.int32).to(device),
            ends=torch.tensor(en, dtype=torch.int32).to(device),
            context_lens=torch.tensor(en, dtype=torch.int32).to(device),
            key=torch.randn(n, H, d, generator=g).to(device),
            value=torch.randn(n, H, d, generator=g).to(device),
            q=torch.randn(2, Hq, d, generator=g).to(device),
        ))
    k0 = torch.zeros(cfg.num_blocks, bs, H, d).to(device)
    v0 = torch.zeros(cfg.num_blocks, bs, H, d).to(device)
    return TinyTrace(cfg=cfg, steps=steps, k_cache0=k0, v_cache0=v0)


@dataclass
class BatchSnapshot:
    """A decode batch's cache described as a CSR block-paged snapshot (one per
    role over the same index buffers): block_table concatenates each
    sequence's ceil(ctx / bs) block ids, seq_ptr delimits the slices and
    token_ptr the sequences' rows of the logical [total_tokens, Hkv, d]."""
    block_table: torch.Tensor  # int32 [nnz]
    seq_ptr: torch.Tensor      # int32 [B+1]
    token_ptr: torch.Tensor    # int64 [B+1]
    total_tokens: int
    nnz: int


def decode_batch_snapshot(batch: DecodeBatch) -> BatchSnapshot:
    bs = batch.cfg.block_size
    ctx = batch.context_lens.cpu().to(torch.int64)
    tables = batch.block_tables.cpu()
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    ids = [tables[b, :n] for b, n in enumerate(nblk)]
    block_table = torch.cat(ids) if ids else torch.zeros(0, dtype=torch.int32)
    seq_ptr = torch.zeros(len(nblk) + 1, dtype=torch.int64)
    seq_ptr[1:] = torch.cumsum(torch.tensor(nblk, dtype=torch.int64), 0)
    token_ptr = torch.zeros(len(nblk) + 1, dtype=torch.int64)
    token_ptr[1:] = torch.cumsum(ctx, 0)
    dev = batch.block_tables.device
    return BatchSnapshot(block_table=block_table.to(torch.int32).to(dev), seq_ptr=seq_ptr.to(torch.int32).to(dev),
                         token_ptr=token_ptr.to(dev), total_tokens=int(token_ptr[-1]), nnz=int(seq_ptr[-1]))
