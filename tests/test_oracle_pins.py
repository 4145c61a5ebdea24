"""Pins for the CPU oracle: each oracle function is checked against something
other than itself -- values the pages print, library routines, closed forms,
special cases and brute force on tiny inputs.

Sources: "Paged KV Cache - AI infra interview lesson" (Walk the Shapes First;
Step 1: slot_mapping and store_kvcache; Step 2: paged_attention_decode;
Common Pitfalls) and "Block-Paged KV Cache" (Element lookup through the block
table; Validating the storage invariants).
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import ROOT, load_golden


# --------------------------------------------------------------------------- widening
def test_widen_f16_exhaustive_matches_numpy(orc):
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.widen_f16(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_widen_bf16_exhaustive_matches_torch(orc):
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    want = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.widen_bf16(int(b) & 0xFFFF) for b in bits.tolist()])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# --------------------------------------------------------------------------- slot mapping
def test_slot_mapping_printed_example(orc):
    g = load_golden("slot_mapping_walk.json")
    slots, err = orc.compute_slot_mapping([g["block_table"]], [g["start"]], [g["end"]],
                                          g["block_size"], num_blocks=8)
    assert err == 0
    assert slots.tolist() == g["slots"]


def _range_form(block_table, start, end, bs):
    """The page's second form: one range per block; the first block may start
    mid-block and the last may be partial (written independently here)."""
    out = []
    if start >= end:
        return out
    first, last = start // bs, (end - 1) // bs
    for blk in range(first, last + 1):
        lo = start - blk * bs if blk == first else 0
        hi = end - blk * bs if blk == last else bs
        out.extend(block_table[blk] * bs + j for j in range(lo, hi))
    return out


@pytest.mark.parametrize("bs", [4, 16, 256])
def test_slot_mapping_equals_range_form(orc, bs):
    bt = [7, 2, 5]
    for start, end in [(0, 2 * bs + 2), (bs // 2 + 1, 2 * bs + 1), (bs, 2 * bs), (3, 3)]:
        slots, err = orc.compute_slot_mapping([bt], [start], [end], bs, num_blocks=8)
        assert err == 0
        assert slots.tolist() == _range_form(bt, start, end, bs)


def test_slot_mapping_concatenates_sequences_and_walk_trace(orc):
    g = load_golden("walk_trace.json")
    tables = [
        [[7, 2, -1], [5, -1, -1]],
        [[7, 2, -1], [5, -1, -1]],
        [[7, 2, -1], [5, 0, -1]],
    ]
    spans = [([0, 0], [6, 3]), ([6, 3], [7, 4]), ([7, 4], [8, 5])]
    for step, bt, (st, en) in zip(g["derived_by_the_page_rules"]["steps"], tables, spans):
        slots, err = orc.compute_slot_mapping(bt, st, en, 4, num_blocks=8)
        assert err == 0
        assert slots.tolist() == step["slots"]
    assert g["derived_by_the_page_rules"]["steps"][0]["slots"][:6] == \
        g["printed_on_page"]["A_prefill"]


def test_decode_slot_pitfall(orc):
    # After appending, A has len 7; the new token sits at position len-1 = 6.
    # The pitfall (last block id * bs + tokens now in the last block) lands at 11.
    row = [7, 2, -1]
    assert orc.slot_of_position(row, 6, 4) == 10
    assert 2 * 4 + 3 == 11 != orc.slot_of_position(row, 6, 4)


def test_slot_mapping_errors_give_minus_one(orc):
    # position 4 needs logical block 1, which is -1; block id 9 >= num_blocks 8
    slots, err = orc.compute_slot_mapping([[7, -1], [9, -1]], [3, 0], [5, 1], 4, num_blocks=8)
    assert slots.tolist() == [31, -1, -1]
    assert err == 2


# --------------------------------------------------------------------------- store_kvcache
@pytest.mark.parametrize("bs", [4, 16, 256])
def test_store_skips_padding_slot(orc, bs):
    """The page's check: slot 1 set to -1 stays zero; exactly n-1 rows written."""
    g = torch.Generator().manual_seed(bs)
    bt, H, d, n = [7, 2, 5], 2, 4, 2 * bs + 2
    kc, vc = torch.zeros(8, bs, H, d), torch.zeros(8, bs, H, d)
    key, value = torch.randn(n, H, d, generator=g), torch.randn(n, H, d, generator=g)
    slots = torch.tensor(_range_form(bt, 0, n, bs), dtype=torch.int32)
    slots[1] = -1
    kc2, vc2, err = orc.store_kvcache(key, value, kc, vc, slots)
    assert err == 0
    for p in range(n):
        wk = torch.zeros(H, d) if p == 1 else key[p]
        wv = torch.zeros(H, d) if p == 1 else value[p]
        assert torch.equal(kc2[bt[p // bs], p % bs], wk)
        assert torch.equal(vc2[bt[p // bs], p % bs], wv)
    assert int((kc2.abs().sum((-1, -2)) != 0).sum()) == n - 1


def test_store_round_trip_bit_exact_bf16(orc):
    g = torch.Generator().manual_seed(1)
    nb, bs, H, d, n = 6, 16, 2, 8, 40
    kc = torch.randn(nb, bs, H, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(nb, bs, H, d, generator=g).to(torch.bfloat16)
    key = torch.randn(n, H, d, generator=g).to(torch.bfloat16)
    value = torch.randn(n, H, d, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    kc2, vc2, err = orc.store_kvcache(key, value, kc, vc, slots)
    assert err == 0
    flat_k, flat_v = kc2.view(-1, H, d), vc2.view(-1, H, d)
    assert torch.equal(flat_k[slots.long()].view(torch.int16), key.view(torch.int16))
    assert torch.equal(flat_v[slots.long()].view(torch.int16), value.view(torch.int16))
    untouched = torch.ones(nb * bs, dtype=torch.bool)
    untouched[slots.long()] = False
    assert torch.equal(flat_k[untouched].view(torch.int16),
                       kc.view(-1, H, d)[untouched].view(torch.int16))


def test_store_out_of_range_slot_is_counted_and_skipped(orc):
    kc, vc = torch.zeros(2, 4, 1, 4), torch.zeros(2, 4, 1, 4)
    key = torch.ones(3, 1, 4)
    kc2, _, err = orc.store_kvcache(key, key, kc, vc, torch.tensor([0, 8, -7], dtype=torch.int32))
    assert err == 2
    assert int((kc2.abs().sum((-1, -2)) != 0).sum()) == 1


# --------------------------------------------------------------------------- attention
def _paged_case(bs, Hq, Hkv, d, lens, nb, seed, dtype=torch.float32):
    """Contiguous K/V per sequence written into a garbage-filled pool through a
    random free list, -1 padded tables (the page's Step 2 test recipe)."""
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(nb, bs, Hkv, d, generator=g).to(dtype)
    vc = torch.randn(nb, bs, Hkv, d, generator=g).to(dtype)
    free = torch.randperm(nb, generator=g).tolist()
    tables, Ks, Vs = [], [], []
    for L in lens:
        bt = [free.pop() for _ in range((L + bs - 1) // bs)]
        K = torch.randn(L, Hkv, d, generator=g).to(dtype)
        V = torch.randn(L, Hkv, d, generator=g).to(dtype)
        for p in range(L):
            kc[bt[p // bs], p % bs] = K[p]
            vc[bt[p // bs], p % bs] = V[p]
        tables.append(bt)
        Ks.append(K)
        Vs.append(V)
    M = max(1, max(len(t) for t in tables))
    block_tables = torch.tensor([t + [-1] * (M - len(t)) for t in tables], dtype=torch.int32)
    q = torch.randn(len(lens), Hq, d, generator=g).to(dtype)
    return q, kc, vc, block_tables, torch.tensor(lens, dtype=torch.int32), Ks, Vs


def _sdpa_reference(q, Ks, Vs, Hq, Hkv, scale):
    outs = []
    for b in range(q.shape[0]):
        K = Ks[b].double().repeat_interleave(Hq // Hkv, 1).transpose(0, 1)
        V = Vs[b].double().repeat_interleave(Hq // Hkv, 1).transpose(0, 1)
        outs.append(F.scaled_dot_product_attention(q[b].double()[:, None], K, V,
                                                   scale=scale)[:, 0])
    return torch.stack(outs)


@pytest.mark.parametrize("bs", [4, 16, 256])
def test_attention_matches_sdpa_on_contiguous_kv(orc, bs):
    Hq, Hkv, d, nb = 4, 2, 8, 12
    lens = [1, bs, 2 * bs + 3]
    q, kc, vc, bt, cl, Ks, Vs = _paged_case(bs, Hq, Hkv, d, lens, nb, seed=bs)
    out, err = orc.paged_attention_decode(q, kc, vc, bt, cl, d ** -0.5)
    assert err == 0
    ref = _sdpa_reference(q, Ks, Vs, Hq, Hkv, d ** -0.5)
    torch.testing.assert_close(out, ref, atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (8, 1)])
def test_attention_half_types_match_sdpa(orc, dtype, Hq, Hkv):
    bs, d = 16, 32
    lens = [5, 16, 40, 77]
    q, kc, vc, bt, cl, Ks, Vs = _paged_case(bs, Hq, Hkv, d, lens, 24, seed=Hq * 10 + Hkv, dtype=dtype)
    out, err = orc.paged_attention_decode(q, kc, vc, bt, cl, 0.3)
    assert err == 0
    ref = _sdpa_reference(q, Ks, Vs, Hq, Hkv, 0.3)
    torch.testing.assert_close(out, ref, atol=1e-12, rtol=1e-12)


def test_attention_gqa_mapping_is_integer_division(orc):
    """Query head h reads KV head h // (Hq/Hkv): give each KV head a constant V
    row equal to its index and check which one every query head sees."""
    bs, Hq, Hkv, d, L = 4, 8, 4, 4, 7
    g = torch.Generator().manual_seed(3)
    kc = torch.randn(2, bs, Hkv, d, generator=g)
    vc = torch.zeros(2, bs, Hkv, d)
    for h in range(Hkv):
        vc[:, :, h, :] = float(h)
    q = torch.randn(1, Hq, d, generator=g)
    out, _ = orc.paged_attention_decode(q, kc, vc, torch.tensor([[0, 1]], dtype=torch.int32),
                                        torch.tensor([L], dtype=torch.int32), 1.0)
    for h in range(Hq):
        want = torch.full((d,), float(h // (Hq // Hkv)), dtype=torch.float64)
        torch.testing.assert_close(out[0, h], want, atol=1e-14, rtol=0)


def test_attention_single_token_returns_v_row_exactly(orc):
    bs, Hq, Hkv, d = 16, 4, 2, 8
    g = torch.Generator().manual_seed(4)
    kc, vc = torch.randn(3, bs, Hkv, d, generator=g), torch.randn(3, bs, Hkv, d, generator=g)
    q = torch.randn(1, Hq, d, generator=g) * 50
    out, _ = orc.paged_attention_decode(q, kc, vc, torch.tensor([[2, -1]], dtype=torch.int32),
                                        torch.tensor([1], dtype=torch.int32), 0.35)
    for h in range(Hq):
        assert torch.equal(out[0, h], vc[2, 0, h // 2].double())


def test_attention_constant_v_and_masked_tail(orc):
    """Constant V rows give V back whatever the scores; NaN in the tail of the
    last block and in unreferenced blocks must never reach the output."""
    bs, Hq, Hkv, d, L = 4, 2, 1, 4, 6
    g = torch.Generator().manual_seed(5)
    kc = torch.full((4, bs, Hkv, d), float("nan"))
    vc = torch.full((4, bs, Hkv, d), float("nan"))
    kc[3, :], kc[1, :2] = torch.randn(bs, Hkv, d, generator=g), torch.randn(2, Hkv, d, generator=g)
    vc[3, :], vc[1, :2] = 2.5, 2.5
    q = torch.randn(1, Hq, d, generator=g)
    out, _ = orc.paged_attention_decode(q, kc, vc, torch.tensor([[3, 1, -1]], dtype=torch.int32),
                                        torch.tensor([L], dtype=torch.int32), 0.5)
    assert not torch.isnan(out).any()
    torch.testing.assert_close(out, torch.full_like(out, 2.5), atol=1e-14, rtol=0)


def test_attention_softmax_closed_form_two_tokens(orc):
    """Two tokens: out = V0 + (V1 - V0) * sigmoid(s1 - s0)."""
    d = 4
    kc = torch.zeros(1, 4, 1, d)
    vc = torch.zeros(1, 4, 1, d)
    kc[0, 0, 0] = torch.tensor([1.0, 0.0, 0.0, 0.0])
    kc[0, 1, 0] = torch.tensor([0.0, 2.0, 0.0, 0.0])
    vc[0, 0, 0] = torch.tensor([1.0, 2.0, 3.0, 4.0])
    vc[0, 1, 0] = torch.tensor([-1.0, 0.5, 0.0, 8.0])
    q = torch.tensor([[[0.75, -0.5, 3.0, 1.0]]])
    out, _ = orc.paged_attention_decode(q, kc, vc, torch.tensor([[0]], dtype=torch.int32),
                                        torch.tensor([2], dtype=torch.int32), 0.8)
    s0, s1 = 0.8 * 0.75, 0.8 * (-1.0)
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    want = vc[0, 0, 0].double() + (vc[0, 1, 0].double() - vc[0, 0, 0].double()) * w1
    torch.testing.assert_close(out[0, 0], want, atol=1e-15, rtol=0)


def test_attention_empty_context_and_bad_block(orc):
    bs, d = 4, 4
    g = torch.Generator().manual_seed(6)
    kc, vc = torch.randn(3, bs, 1, d, generator=g), torch.randn(3, bs, 1, d, generator=g)
    q = torch.randn(2, 1, d, generator=g)
    bt = torch.tensor([[0, -1], [1, 7]], dtype=torch.int32)   # 7 >= num_blocks
    out, err = orc.paged_attention_decode(q, kc, vc, bt, torch.tensor([0, 6], dtype=torch.int32), 1.0)
    assert torch.equal(out[0], torch.zeros(1, d, dtype=torch.float64))
    assert err == 1
    # the bad block's tokens are dropped: the same as attending over block 1 only
    want, _ = orc.paged_attention_decode(q[1:], kc, vc, torch.tensor([[1]], dtype=torch.int32),
                                         torch.tensor([4], dtype=torch.int32), 1.0)
    torch.testing.assert_close(out[1], want[0], atol=1e-15, rtol=0)


# --------------------------------------------------------------------------- CSR snapshot
def test_decode_step_walk_appends_at_ctx_minus_one_and_attends(orc):
    """The walk of "Walk the Shapes First": after the prefill (A: 6 tokens in
    blocks [7, 2], B: 3 tokens in block [5]), decode step 1 appends A's token at
    slot 10 and B's at slot 23 (the golden trace), then attends over 7 and 4
    tokens; the output equals SDPA over the same rows stored contiguously."""
    g = torch.Generator().manual_seed(5)
    bs, Hkv, Hq, d = 4, 2, 4, 4
    kc, vc = torch.randn(8, bs, Hkv, d, generator=g), torch.randn(8, bs, Hkv, d, generator=g)
    tables = torch.tensor([[7, 2], [5, -1]], dtype=torch.int32)
    key, value = torch.randn(2, Hkv, d, generator=g), torch.randn(2, Hkv, d, generator=g)
    q = torch.randn(2, Hq, d, generator=g)
    cl = torch.tensor([7, 4], dtype=torch.int32)
    out, kc2, vc2, err = orc.decode_step(q, key, value, kc, vc, tables, cl, 0.5)
    assert err == 0
    want = load_golden("walk_trace.json")["derived_by_the_page_rules"]["steps"][1]["slots"]
    flat_k, flat_v = kc2.reshape(-1, Hkv, d), vc2.reshape(-1, Hkv, d)
    for b, slot in enumerate(want):
        assert torch.equal(flat_k[slot], key[b]) and torch.equal(flat_v[slot], value[b])
    changed = (kc2 != kc).reshape(-1, Hkv * d).any(1).nonzero().reshape(-1).tolist()
    assert changed == sorted(want)
    # contiguous K/V by hand: A = block 7 rows 0-3, block 2 rows 0-1, then its new row;
    # B = block 5 rows 0-2, then its new row
    Ks = [torch.cat([kc[7], kc[2, :2], key[0:1]]), torch.cat([kc[5, :3], key[1:2]])]
    Vs = [torch.cat([vc[7], vc[2, :2], value[0:1]]), torch.cat([vc[5, :3], value[1:2]])]
    torch.testing.assert_close(out, _sdpa_reference(q, Ks, Vs, Hq, Hkv, 0.5), atol=1e-12, rtol=1e-12)


def test_element_offset_printed_example_and_alias(orc):
    g = load_golden("element_offset_example.json")
    args = (g["page_size"], g["num_pages"], g["num_heads"], g["head_dim"], g["block_table"],
            g["seq_ptr"])
    for idx in (torch.int32, torch.int64):
        for lk in g["lookups"]:
            assert orc.element_offset(lk["seq"], lk["token"], lk["head"], lk["dim"], *args,
                                      index_dtype=idx) == lk["flat"]
        for a, b in g["aliased"]:
            oa = orc.element_offset(a["seq"], a["token"], a["head"], a["dim"], *args, index_dtype=idx)
            ob = orc.element_offset(b["seq"], b["token"], b["head"], b["dim"], *args, index_dtype=idx)
            assert oa == ob >= 0


def test_element_offset_closed_form_and_errors(orc):
    ps, npg, H, d = 4, 5, 2, 8
    sp, bt = [0, 2, 3], [3, 1, 4]
    for s, lo, hi in ((0, 0, 2), (1, 2, 3)):
        for t in range((hi - lo) * ps):
            for h in range(H):
                for i in range(d):
                    phys = bt[lo + t // ps]
                    want = phys * ps * H * d + (t % ps) * H * d + h * d + i
                    assert orc.element_offset(s, t, h, i, ps, npg, H, d, bt, sp) == want
    assert orc.element_offset(2, 0, 0, 0, ps, npg, H, d, bt, sp) == -1     # seq out of range
    assert orc.element_offset(1, 4, 0, 0, ps, npg, H, d, bt, sp) == -1     # beyond the slice
    assert orc.element_offset(0, 0, 2, 0, ps, npg, H, d, bt, sp) == -1     # head out of range
    assert orc.element_offset(0, 0, 0, 8, ps, npg, H, d, bt, sp) == -1     # dim out of range
    assert orc.element_offset(1, 0, 0, 0, ps, 4, H, d, bt, sp) == -1       # page 4 >= num_pages


def test_validator_printed_cases(orc):
    g = load_golden("validator_cases.json")
    for c in g["cases"]:
        for idx in (torch.int32, torch.int64):
            code = orc.validate_index_buffers(c["seq_ptr"], c["block_table"], g["num_pages"], idx)
            assert (code == 0) == c["valid"], c["note"]


def test_validator_each_invariant(orc):
    assert orc.validate_index_buffers([1, 2, 3], [0, 1, 0], 5) == 1   # seq_ptr[0] != 0
    assert orc.validate_index_buffers([0, 2, 1], [0, 1, 0], 5) == 2   # decreasing
    assert orc.validate_index_buffers([0, 2, 2], [0, 1, 0], 5) == 3   # last != len(block_table)
    assert orc.validate_index_buffers([0, 2, 3], [0, 1, 9], 5) == 4   # page out of range


def test_unpack_identity_table_is_a_reshape(orc):
    g = torch.Generator().manual_seed(7)
    npg, ps, H, d = 6, 4, 2, 8
    pool = torch.randn(npg, ps, H, d, generator=g).to(torch.bfloat16)
    out, err = orc.unpack_block_paged(pool, list(range(npg)), [0, npg], [0, npg * ps])
    assert err == 0
    assert torch.equal(out.view(torch.int16), pool.reshape(npg * ps, H, d).view(torch.int16))


def test_unpack_printed_layout_brute_force_and_alias(orc):
    """The page's snapshot (seq_ptr [0,2,3], block_table [0,1,0], page_size 4,
    H 2, d 8, logical shape [9, 2, 8]), read with both 5+4 and 8+1 splits."""
    g = torch.Generator().manual_seed(8)
    pool = torch.randn(5, 4, 2, 8, generator=g)
    for lens in ([5, 4], [8, 1]):
        tp = [0, lens[0], lens[0] + lens[1]]
        for idx in (torch.int32, torch.int64):
            out, err = orc.unpack_block_paged(pool, [0, 1, 0], [0, 2, 3], tp, index_dtype=idx)
            assert err == 0 and out.shape == (9, 2, 8)
            pages = {0: [0, 1], 1: [0]}
            for s in (0, 1):
                for t in range(lens[s]):
                    assert torch.equal(out[tp[s] + t], pool[pages[s][t // 4], t % 4])
            # seq 1 token 0 aliases seq 0 token 0
            assert torch.equal(out[tp[1]], out[0])


def test_unpack_missing_page_is_zero_and_counted(orc):
    pool = torch.ones(2, 2, 1, 4)
    out, err = orc.unpack_block_paged(pool, [1], [0, 1], [0, 3])   # token 2 needs a 2nd page
    assert torch.equal(out[:2], pool[1])
    assert torch.equal(out[2], torch.zeros(1, 4)) and err == 4


# --------------------------------------------------------------------------- fp8 (E4M3) cache
def test_e4m3_decode_exhaustive_matches_torch(orc):
    """Every one of the 256 codes against torch's float8_e4m3fn."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(torch.float8_e4m3fn).double()
    got = torch.tensor([orc.e4m3_decode(c) for c in range(256)], dtype=torch.float64)
    nan = torch.isnan(want)
    assert torch.equal(nan, torch.isnan(got)) and nan.sum() == 2  # S.1111.111
    assert torch.equal(got[~nan], want[~nan])
    assert orc.e4m3_decode(0x7E) == 448.0 and orc.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_rounds_to_nearest_even(orc):
    """Against torch's cast (round to nearest even) on every representable
    value, every midpoint and its float32 neighbours, and random magnitudes
    from the subnormal range to 448."""
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    fin = vals[~torch.isnan(vals)].unique()
    pos = fin[fin >= 0]
    mids = (pos[1:] + pos[:-1]) / 2
    g = torch.Generator().manual_seed(8)
    rnd = torch.exp(torch.empty(20000).uniform_(-10 * 0.6931, 8.8 * 0.6931, generator=g))
    xs = torch.cat([fin, mids, torch.nextafter(mids, torch.full_like(mids, 1e9)),
                    torch.nextafter(mids, torch.zeros_like(mids)), rnd, -rnd]).float()
    xs = xs[xs.abs() <= 448]
    want = xs.to(torch.float8_e4m3fn).view(torch.uint8)
    got = torch.tensor([orc.e4m3_encode(float(x)) for x in xs], dtype=torch.uint8)
    assert torch.equal(got, want)


def test_e4m3_encode_saturates_and_keeps_nan(orc):
    for x, code in [(448.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E),
                    (-1e30, 0xFE), (float("-inf"), 0xFE), (float("nan"), 0x7F), (-0.0, 0x80),
                    (2.0 ** -10, 0x00), (1.5 * 2.0 ** -9, 0x02)]:
        assert orc.e4m3_encode(x) == code, x


def test_quantize_and_store_fp8_match_a_torch_restatement(orc):
    """Per (block, head) s = max|x| / 448, codes = x / s cast to E4M3 (binary32
    division), against torch; the store writes the same codes at the slots."""
    g = torch.Generator().manual_seed(9)
    nb, bs, H, d = 5, 4, 2, 8
    cache = (torch.randn(nb, bs, H, d, generator=g) * 3).to(torch.bfloat16)
    cache[2, :, 1] = 0  # an all-zero (block, head): scale 0, codes +0
    codes, scales = orc.quantize_kvcache_fp8(cache)
    amax = cache.float().abs().amax(dim=(1, 3))
    assert torch.equal(scales, amax / 448.0)
    safe = torch.where(scales == 0, torch.ones_like(scales), scales)
    want = (cache.float() / safe[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    want[2, :, 1] = 0
    assert torch.equal(codes, want)
    # the store: tokens 0..2 at slots 9, -1, 17 with the blocks' scales
    key = (torch.randn(3, H, d, generator=g) * 2).to(torch.bfloat16)
    value = (torch.randn(3, H, d, generator=g) * 2).to(torch.bfloat16)
    slots = torch.tensor([9, -1, 17], dtype=torch.int32)
    kc, vc, err = orc.store_kvcache_fp8(key, value, codes, codes, scales, scales, slots)
    assert err == 0
    for i, slot in ((0, 9), (2, 17)):  # slot 9 is block 2, whose head 1 has scale 0
        blk = slot // bs
        x = (key[i].float() / safe[blk][:, None]).clamp(-448, 448)  # saturation, then RN-even
        want_k = x.to(torch.float8_e4m3fn).view(torch.uint8)
        want_k[scales[blk] == 0] = 0
        assert torch.equal(kc.reshape(-1, H, d)[slot], want_k)
    assert torch.equal(kc.reshape(-1, H, d)[[s for s in range(nb * bs) if s not in (9, 17)]],
                       codes.reshape(-1, H, d)[[s for s in range(nb * bs) if s not in (9, 17)]])


def test_attention_fp8_matches_sdpa_on_dequantized_kv(orc):
    """The fp8 attention equals SDPA (binary64) over K/V dequantized as
    scale * decode(code) and stored contiguously."""
    bs, Hq, Hkv, d, nb = 4, 4, 2, 8, 12
    q, kc, vc, bt, cl, _, _ = _paged_case(bs, Hq, Hkv, d, [1, bs, 2 * bs + 3], nb, seed=10)
    kq, ks = orc.quantize_kvcache_fp8(kc)
    vq, vs = orc.quantize_kvcache_fp8(vc)
    out, err = orc.paged_attention_decode_fp8(q, kq, vq, ks, vs, bt, cl, d ** -0.5)
    assert err == 0
    dk = kq.view(torch.float8_e4m3fn).double() * ks.double()[:, None, :, None]
    dv = vq.view(torch.float8_e4m3fn).double() * vs.double()[:, None, :, None]
    Ks, Vs = [], []
    for b in range(3):
        n = int(cl[b])
        rows = [(int(bt[b, t // bs]), t % bs) for t in range(n)]
        Ks.append(torch.stack([dk[p, o] for p, o in rows]))
        Vs.append(torch.stack([dv[p, o] for p, o in rows]))
    torch.testing.assert_close(out, _sdpa_reference(q, Ks, Vs, Hq, Hkv, d ** -0.5), atol=1e-12, rtol=1e-12)


def _int8_restatement(y):
    """torch's round (half to even) and clamp: the int8 code of binary32 values y."""
    r = torch.round(y.float()).clamp(-127, 127)
    return torch.where(torch.isnan(y), torch.zeros_like(r), r).to(torch.int8)


def test_int8_encode_rounds_half_even_and_clamps(orc):
    halves = torch.arange(-130, 131, dtype=torch.float32) + 0.5
    g = torch.Generator().manual_seed(11)
    rnd = torch.empty(20000).uniform_(-140, 140, generator=g)
    xs = torch.cat([halves, torch.nextafter(halves, torch.full_like(halves, 1e9)),
                    torch.nextafter(halves, torch.full_like(halves, -1e9)), rnd,
                    torch.tensor([0.0, -0.0, 1e30, -1e30, float("inf"), float("-inf"), float("nan")])])
    got = torch.tensor([orc.int8_encode(float(x)) for x in xs], dtype=torch.int8)
    assert torch.equal(got, _int8_restatement(xs))
    for x, code in [(0.5, 0), (1.5, 2), (2.5, 2), (-2.5, -2), (126.5, 126), (127.5, 127), (-127.5, -127),
                    (float("nan"), 0)]:
        assert orc.int8_encode(x) == code, x


def test_quantize_and_store_int8_match_a_torch_restatement(orc):
    """Per (block, head) s = max|x| / 127, codes = round(x / s) (binary32
    division, ties to even) clamped to [-127, 127], against torch; the store
    writes the same codes at the slots."""
    g = torch.Generator().manual_seed(12)
    nb, bs, H, d = 5, 4, 2, 8
    cache = (torch.randn(nb, bs, H, d, generator=g) * 3).to(torch.float16)
    cache[2, :, 1] = 0  # an all-zero (block, head): scale 0, codes 0
    codes, scales = orc.quantize_kvcache_int8(cache)
    amax = cache.float().abs().amax(dim=(1, 3))
    assert codes.dtype == torch.int8 and torch.equal(scales, amax / 127.0)
    safe = torch.where(scales == 0, torch.ones_like(scales), scales)
    want = _int8_restatement(cache.float() / safe[:, None, :, None])
    want[2, :, 1] = 0
    assert torch.equal(codes, want)
    assert codes.abs().amax() == 127  # each block's largest element maps to +-127
    key = (torch.randn(3, H, d, generator=g) * 4).to(torch.float16)  # some beyond 127 s: clamped
    value = (torch.randn(3, H, d, generator=g) * 2).to(torch.float16)
    slots = torch.tensor([9, -1, 17], dtype=torch.int32)
    kc, vc, err = orc.store_kvcache_int8(key, value, codes, codes, scales, scales, slots)
    assert err == 0
    for i, slot in ((0, 9), (2, 17)):  # slot 9 is block 2, whose head 1 has scale 0
        blk = slot // bs
        want_k = _int8_restatement(key[i].float() / safe[blk][:, None])
        want_k[scales[blk] == 0] = 0
        assert torch.equal(kc.reshape(-1, H, d)[slot], want_k)
    others = [s for s in range(nb * bs) if s not in (9, 17)]
    assert torch.equal(kc.reshape(-1, H, d)[others], codes.reshape(-1, H, d)[others])


def test_attention_int8_matches_sdpa_on_dequantized_kv(orc):
    """The int8 attention equals SDPA (binary64) over K/V dequantized as
    scale * code and stored contiguously."""
    bs, Hq, Hkv, d, nb = 4, 4, 2, 8, 12
    q, kc, vc, bt, cl, _, _ = _paged_case(bs, Hq, Hkv, d, [1, bs, 2 * bs + 3], nb, seed=13)
    kq, ks = orc.quantize_kvcache_int8(kc)
    vq, vs = orc.quantize_kvcache_int8(vc)
    out, err = orc.paged_attention_decode_int8(q, kq, vq, ks, vs, bt, cl, d ** -0.5)
    assert err == 0
    dk = kq.double() * ks.double()[:, None, :, None]
    dv = vq.double() * vs.double()[:, None, :, None]
    Ks, Vs = [], []
    for b in range(3):
        n = int(cl[b])
        rows = [(int(bt[b, t // bs]), t % bs) for t in range(n)]
        Ks.append(torch.stack([dk[p, o] for p, o in rows]))
        Vs.append(torch.stack([dv[p, o] for p, o in rows]))
    torch.testing.assert_close(out, _sdpa_reference(q, Ks, Vs, Hq, Hkv, d ** -0.5), atol=1e-12, rtol=1e-12)


# --------------------------------------------------------------------------- varlen / chunked prefill
def _prefill_case(bs, Hq, Hkv, d, spans, nb, seed, dtype=torch.float32):
    """spans: (start, n) per sequence; contiguous K/V of length start + n are
    scattered into random blocks; q holds the n queries of each sequence."""
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(nb, bs, Hkv, d, generator=g).to(dtype)
    vc = torch.randn(nb, bs, Hkv, d, generator=g).to(dtype)
    free = torch.randperm(nb, generator=g).tolist()
    tables, Ks, Vs = [], [], []
    for start, n in spans:
        L = start + n
        bt = [free.pop() for _ in range((L + bs - 1) // bs)]
        K, V = torch.randn(L, Hkv, d, generator=g).to(dtype), torch.randn(L, Hkv, d, generator=g).to(dtype)
        for p in range(L):
            kc[bt[p // bs], p % bs], vc[bt[p // bs], p % bs] = K[p], V[p]
        tables.append(bt)
        Ks.append(K)
        Vs.append(V)
    M = max(1, max(len(t) for t in tables))
    block_tables = torch.tensor([t + [-1] * (M - len(t)) for t in tables], dtype=torch.int32)
    starts = torch.tensor([s for s, _ in spans], dtype=torch.int32)
    cu = torch.zeros(len(spans) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor([n for _, n in spans]), 0)
    q = torch.randn(int(cu[-1]), Hq, d, generator=g).to(dtype)
    return q, kc, vc, block_tables, starts, cu, Ks, Vs


@pytest.mark.parametrize("bs", [4, 16])
def test_prefill_matches_sdpa_with_causal_mask(orc, bs):
    """Against SDPA (binary64) on the same K/V stored contiguously, with the
    mask key <= query position, for a plain prefill, chunks after a cached
    prefix, a single new token and block-straddling spans."""
    Hq, Hkv, d = 4, 2, 8
    spans = [(0, 2 * bs + 3), (bs + 1, 5), (3 * bs, bs), (7, 1), (0, 1)]
    q, kc, vc, bt, st, cu, Ks, Vs = _prefill_case(bs, Hq, Hkv, d, spans, 40, seed=bs + 60)
    out, err = orc.paged_attention_prefill(q, kc, vc, bt, st, cu, d ** -0.5)
    assert err == 0
    for b, (start, n) in enumerate(spans):
        L = start + n
        K = Ks[b].double().repeat_interleave(Hq // Hkv, 1).transpose(0, 1)  # [Hq, L, d]
        V = Vs[b].double().repeat_interleave(Hq // Hkv, 1).transpose(0, 1)
        Q = q[int(cu[b]):int(cu[b + 1])].double().transpose(0, 1)            # [Hq, n, d]
        mask = torch.arange(L)[None, :] <= (start + torch.arange(n))[:, None]
        ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=d ** -0.5).transpose(0, 1)
        torch.testing.assert_close(out[int(cu[b]):int(cu[b + 1])], ref, atol=1e-12, rtol=1e-12)


def test_prefill_last_query_equals_decode(orc):
    """The last new token of a sequence sees its whole context: the prefill
    row equals the (separately pinned) decode attention over start + n tokens."""
    bs, Hq, Hkv, d = 16, 8, 2, 16
    spans = [(40, 9), (0, 33), (16, 16)]
    q, kc, vc, bt, st, cu, _, _ = _prefill_case(bs, Hq, Hkv, d, spans, 30, seed=61, dtype=torch.bfloat16)
    out, err = orc.paged_attention_prefill(q, kc, vc, bt, st, cu, 0.3)
    last = cu[1:] - 1
    dec, derr = orc.paged_attention_decode(q[last], kc, vc, bt, st + (cu[1:] - cu[:-1]), 0.3)
    assert err == 0 == derr
    torch.testing.assert_close(out[last], dec, atol=1e-12, rtol=1e-12)


def test_prefill_bad_inputs_zero_rows_and_count(orc):
    bs, Hq, Hkv, d = 4, 2, 1, 4
    q, kc, vc, bt, st, cu, _, _ = _prefill_case(bs, Hq, Hkv, d, [(2, 3), (0, 4)], 8, seed=62)
    bt2 = bt.clone()
    bt2[1, 0] = 99  # sequence 1's only block is outside the pool: all its keys dropped
    out, err = orc.paged_attention_prefill(q, kc, vc, bt2, st, cu, 0.5)
    assert err == 1 and torch.count_nonzero(out[3:]) == 0
    st3 = torch.tensor([-1, 0], dtype=torch.int32)  # a negative start: zero rows, counted
    out, err = orc.paged_attention_prefill(q, kc, vc, bt, st3, cu, 0.5)
    assert err == 1 and torch.count_nonzero(out[:3]) == 0


def test_quantization_compatibility_printed_cases(orc):
    """The page's three printed cases (page_size 4): per-block-affine along
    axis 0 with block_size == page_size fits; block_size 8 does not; per-channel
    along the paged axis does not."""
    g = load_golden("quantization_cases.json")
    for c in g["cases"]:
        code = orc.quantization_compatible(g["scheme_tags"][c["scheme"]], c["axis"], c["block_size"], g["page_size"])
        assert (code == 0) == c["valid"], c["note"]


def test_quantization_compatibility_each_rule(orc):
    assert orc.quantization_compatible(0x03, 1, 4, 4) == 1   # per-block-affine off the paged axis
    assert orc.quantization_compatible(0x03, 0, 2, 4) == 2   # block_size != page_size
    assert orc.quantization_compatible(0x02, 0, 4, 4) == 3   # per-channel on the paged axis
    assert orc.quantization_compatible(0x02, 2, 4, 4) == 0   # per-channel along heads
    assert orc.quantization_compatible(0x01, 0, 1, 4) == 0   # per-tensor
    assert orc.quantization_compatible(0x00, 0, 1, 4) == 0   # none
    assert orc.quantization_compatible(0x07, 0, 4, 4) == 4   # unknown tag


def test_walk_trace_golden_is_what_its_script_derives():
    """walk_trace.json's derived steps are written by tests/golden/make_walk_trace.py,
    which calls only the oracle (allocator model and slot mapping)."""
    import importlib.util

    path = os.path.join(ROOT, "tests", "golden", "make_walk_trace.py")
    spec = importlib.util.spec_from_file_location("_make_walk_trace", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.main(["--check"]) == 0
    steps = load_golden("walk_trace.json")["derived_by_the_page_rules"]["steps"]
    assert steps[0]["slots"][:6] == load_golden("walk_trace.json")["printed_on_page"]["A_prefill"]
