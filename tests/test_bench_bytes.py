"""The benchmark's byte accounting on CPU: the algorithmic bytes its GB/s
figures divide by, checked against brute-force counts over small workloads."""
import torch

import bench
import pkv_workloads as wl


def _row_bytes(cfg):
    return cfg.num_heads * cfg.head_dim * torch.tensor([], dtype=cfg.dtype).element_size()


def test_csr_unique_and_logical_bytes_match_a_brute_force_count():
    """Unique bytes count each (page, row) a sequence reads once; the closed form
    (all tokens minus the aliased prefix's repeats) equals the size of the set of
    (page, row) pairs the CSR index buffers name."""
    cfg = wl.CSR_PREFIX
    snap = wl.csr_snapshot(cfg, seed=3, num_seqs=12, prefix_tokens=64, suffix_hi=70)
    unique, logical, unique_tokens = bench.csr_step_bytes(snap.cfg, snap)
    bt, sp, lens = snap.block_table.tolist(), snap.seq_ptr.tolist(), snap.seq_lens.tolist()
    ps = cfg.page_size
    rows = {(bt[sp[s] + t // ps], t % ps) for s in range(len(lens)) for t in range(lens[s])}
    assert unique_tokens == len(rows)
    row = _row_bytes(cfg)
    T = sum(lens)
    idx = len(bt) * 4 + (len(lens) + 1) * 12
    assert unique["unpack_k"] == T * row + len(rows) * row + idx
    assert logical["unpack_k"] == 2 * T * row + idx
    q_and_out = 2 * len(lens) * cfg.num_heads * cfg.head_dim * 2
    tables = snap.block_tables_2d.numel() * 4 + len(lens) * 4
    assert unique["paged_attention_decode"] == 2 * len(rows) * row + q_and_out + tables
    assert logical["paged_attention_decode"] == 2 * T * row + q_and_out + tables


def test_csr_sub_snapshot_keeps_each_sequences_pages():
    snap = wl.csr_snapshot(wl.CSR_PREFIX, seed=4, num_seqs=10, prefix_tokens=32, suffix_hi=50)
    sub = bench.csr_sub_snapshot(snap, 4, 3)
    sp = snap.seq_ptr.tolist()
    for k in range(3):
        s = 4 + k
        pages = snap.block_table[sp[s]:sp[s + 1]].tolist()
        assert sub.block_table[int(sub.seq_ptr[k]):int(sub.seq_ptr[k + 1])].tolist() == pages
        assert int(sub.token_ptr[k + 1] - sub.token_ptr[k]) == int(snap.seq_lens[s])
    assert sub.total_tokens == int(snap.seq_lens[4:7].sum())


def test_decode_step_bytes_count_every_context_row_once():
    cfg = wl.LONG_GQA_8K
    ctx = torch.tensor([5, 0, 17, 4096], dtype=torch.int32)
    b = bench.step_bytes(cfg, ctx, nnz=1 + 0 + 2 + 256)
    row = cfg.num_kv_heads * cfg.head_dim * 2
    T = int(ctx.sum())
    assert b["paged_attention_decode"] == T * 2 * row + 2 * 4 * cfg.num_q_heads * cfg.head_dim * 2 + 259 * 4 + 4 * 4
    assert b["unpack_k"] == b["unpack_v"] == 2 * T * row + 259 * 4 + 5 * 12


def test_code8_attention_bytes_count_one_byte_per_element_and_the_scales():
    """8-bit (E4M3 / int8) attention bytes: each context row's K and V codes
    once (one byte per element), a K and a V fp32 scale per (table entry, KV
    head), q and out in the query dtype, the table entries and the lengths."""
    cfg = wl.LONG_GQA_8K
    ctx = torch.tensor([5, 0, 17, 4096], dtype=torch.int32)
    nnz = 1 + 0 + 2 + 256
    got = bench.code8_attention_bytes(cfg, ctx, nnz)
    T = int(ctx.sum())
    codes = T * 2 * cfg.num_kv_heads * cfg.head_dim
    q_and_out = 2 * 4 * cfg.num_q_heads * cfg.head_dim * 2
    scales = nnz * cfg.num_kv_heads * 2 * 4
    assert got == codes + q_and_out + nnz * 4 + 4 * 4 + scales
    # half the 16-bit attention's K/V bytes, plus the scales
    b16 = bench.step_bytes(cfg, ctx, nnz)["paged_attention_decode"]
    assert got - scales == b16 - codes
