"""Host-side checks of libpkv.so that need no GPU: every symbol the header
declares is exported, the host validators agree with the pages' printed cases,
and argument checks fail synchronously before any CUDA work is enqueued."""
import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT, load_golden


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    return sorted(set(re.findall(r"PKV_API[^;(]*?\b(pkv_\w+)\s*\(", text)))


def test_header_symbols_are_exported(pkv):
    names = _declared_symbols()
    assert len(names) >= 12
    lib = ctypes.CDLL(pkv.LIBRARY_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) >= {"pkv_compute_slot_mapping", "pkv_store_kvcache", "pkv_paged_attention_decode",
                          "pkv_unpack_block_paged"}


def test_version(pkv):
    assert "sm_103a" in pkv.pkv_version()


def test_validator_printed_cases(pkv):
    g = load_golden("validator_cases.json")
    for c in g["cases"]:
        for idx in (torch.int32, torch.int64):
            if c["valid"]:
                pkv.pkv_validate_index_buffers(c["seq_ptr"], c["block_table"], g["num_pages"], idx)
            else:
                with pytest.raises(pkv.PkvError) as e:
                    pkv.pkv_validate_index_buffers(c["seq_ptr"], c["block_table"], g["num_pages"], idx)
                assert e.value.status == pkv.PKV_ERR_OUT_OF_RANGE


@pytest.mark.parametrize("seq_ptr,block_table", [([1, 2, 3], [0, 1, 0]), ([0, 2, 1], [0, 1, 0]),
                                                  ([0, 2, 2], [0, 1, 0]), ([0, 2, 3], [0, 1, 9])])
def test_validator_rejects_each_invariant(pkv, seq_ptr, block_table):
    with pytest.raises(pkv.PkvError):
        pkv.pkv_validate_index_buffers(seq_ptr, block_table, 5)


def test_element_offset_printed_example(pkv):
    g = load_golden("element_offset_example.json")
    args = (g["page_size"], g["num_pages"], g["num_heads"], g["head_dim"], g["block_table"], g["seq_ptr"])
    for idx in (torch.int32, torch.int64):
        for lk in g["lookups"]:
            assert pkv.pkv_block_paged_element_offset(lk["seq"], lk["token"], lk["head"], lk["dim"], *args,
                                                      index_dtype=idx) == lk["flat"]
        for a, b in g["aliased"]:
            assert pkv.pkv_block_paged_element_offset(a["seq"], a["token"], a["head"], a["dim"], *args) == \
                pkv.pkv_block_paged_element_offset(b["seq"], b["token"], b["head"], b["dim"], *args)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_block_paged_element_offset(1, 4, 0, 0, *args)  # beyond seq 1's single page


def test_element_offset_matches_oracle_everywhere(pkv, orc):
    g = torch.Generator().manual_seed(11)
    ps, npg, H, d = 4, 9, 3, 5
    lens = [7, 1, 12, 4]
    pages = [torch.randint(0, npg, ((n + ps - 1) // ps,), generator=g).tolist() for n in lens]
    seq_ptr = [0]
    for p in pages:
        seq_ptr.append(seq_ptr[-1] + len(p))
    bt = [x for p in pages for x in p]
    for s, n in enumerate(lens):
        for t in range(n + ps):  # includes tokens past the sequence's pages
            for h in range(H):
                for i in range(d):
                    want = orc.element_offset(s, t, h, i, ps, npg, H, d, bt, seq_ptr)
                    if want < 0:
                        with pytest.raises(pkv.PkvError):
                            pkv.pkv_block_paged_element_offset(s, t, h, i, ps, npg, H, d, bt, seq_ptr)
                    else:
                        assert pkv.pkv_block_paged_element_offset(s, t, h, i, ps, npg, H, d, bt, seq_ptr) == want


def test_token_ptr_and_shape_checks(pkv):
    pkv.pkv_validate_token_ptr([0, 5, 9], [0, 2, 3], 4, 9)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_validate_token_ptr([0, 9, 9], [0, 2, 3], 4, 9)   # 9 tokens need 3 pages, seq 0 has 2
    with pytest.raises(pkv.PkvError):
        pkv.pkv_validate_token_ptr([0, 5, 8], [0, 2, 3], 4, 9)   # does not end at total_tokens
    pkv.pkv_validate_block_paged_shape([9, 2, 8], 2, 8)         # the page's rank-3 example
    with pytest.raises(pkv.PkvError):
        pkv.pkv_validate_block_paged_shape([9, 2], 2, 8)        # rank-2 is refused


def test_decode_argument_errors_are_synchronous(pkv):
    lib = pkv._lib
    # Hq not a multiple of Hkv: rejected before anything touches a device.
    st = lib.pkv_paged_attention_decode(None, None, None, None, None, 1, None, 2, 6, 4, 128, 16, 10, 64,
                                        1.0, pkv.PKV_BF16, None, 0, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    assert b"multiple" in lib.pkv_last_error_string()
    st = lib.pkv_paged_attention_decode(None, None, None, None, None, 1, None, 2, 8, 4, 128, 16, 10, 64,
                                        1.0, 7, None, 0, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # NULL pointers with work to do
    st = lib.pkv_paged_attention_decode(None, None, None, None, None, 1, None, 2, 8, 4, 128, 16, 10, 64,
                                        1.0, pkv.PKV_BF16, None, 0, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    # empty batch is a no-op
    st = lib.pkv_paged_attention_decode(None, None, None, None, None, 0, None, 0, 8, 4, 128, 16, 10, 64,
                                        1.0, pkv.PKV_BF16, None, 0, None, None)
    assert st == pkv.PKV_OK
    assert lib.pkv_store_kvcache(None, None, None, None, None, 3, 2, 4, 16, pkv.PKV_F32, None, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_store_kvcache(None, None, None, None, None, 0, 2, 4, 16, pkv.PKV_F32, None, None) == pkv.PKV_OK
    assert lib.pkv_compute_slot_mapping(None, 4, None, None, None, 2, 0, 8, None, 0, None, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_unpack_block_paged(None, None, None, None, 2, None, 1, 1, 4, 5, 2, 8, 9, pkv.PKV_BF16, None,
                                      None) == pkv.PKV_ERR_INVALID_ARG
    # the fused decode step: missing key/value, then the decode checks
    st = lib.pkv_paged_attention_decode_append(None, None, None, None, None, None, None, 1, None, 2, 8, 4, 128, 16,
                                               10, 64, 1.0, pkv.PKV_BF16, None, 0, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG and b"key or value" in lib.pkv_last_error_string()
    st = lib.pkv_paged_attention_decode_append(None, None, 8, 8, None, None, None, 1, None, 2, 6, 4, 128, 16,
                                               10, 64, 1.0, pkv.PKV_BF16, None, 0, None, None)
    assert st == pkv.PKV_ERR_INVALID_ARG and b"multiple" in lib.pkv_last_error_string()
    assert lib.pkv_paged_attention_decode_append(None, None, None, None, None, None, None, 0, None, 0, 8, 4, 128,
                                                 16, 10, 64, 1.0, pkv.PKV_BF16, None, 0, None, None) == pkv.PKV_OK


def test_workspace_size_and_plan(pkv):
    # CUDA-core path: one partition -> no workspace
    assert pkv.pkv_paged_attention_decode_workspace_size(4, 8, 8, 64, 16, 100, torch.float32) == 0
    # tensor-core path, work-balanced schedule (partition 0): room for one piece per (unit, CTA) boundary
    p, n, fast = pkv.pkv_paged_attention_decode_plan(8, 32, 8, 128, 16, 32768, torch.bfloat16)
    assert fast and p == 0
    ws = pkv.pkv_paged_attention_decode_workspace_size(8, 32, 8, 128, 16, 32768, torch.bfloat16)
    units, heads_per_unit = 8 * 2, 16
    assert ws >= (units + 512) * heads_per_unit * (128 * 4 + 8) + 2 * units * 4
    # more than 1024 sequences: tensor-core path with fixed partitions of the context
    p, n, fast = pkv.pkv_paged_attention_decode_plan(2000, 32, 8, 128, 16, 32768, torch.bfloat16)
    assert fast and p % 16 == 0 and p > 0 and n == -(-32768 // p)
    assert not pkv.pkv_paged_attention_decode_plan(2, 4, 2, 8, 4, 64, torch.float32)[2]   # CUDA-core path
    assert not pkv.pkv_paged_attention_decode_plan(2, 32, 2, 128, 16, 64, torch.bfloat16)[2]  # G = 16 > 8
    assert pkv.pkv_paged_attention_decode_workspace_size(2, 6, 4, 128, 16, 64, torch.bfloat16) == 0  # invalid


def test_binding_refuses_cpu_tensors(pkv):
    t = torch.zeros(2, 2, 4)
    with pytest.raises(ValueError):
        pkv.pkv_paged_attention_decode(t, torch.zeros(1, 4, 2, 4), torch.zeros(1, 4, 2, 4),
                                       torch.zeros(2, 1, dtype=torch.int32), torch.ones(2, dtype=torch.int32),
                                       1.0, 4)


def test_prefill_argument_errors_are_synchronous(pkv):
    """The prefill entry rejects bad shapes and alignments before any CUDA call
    (the pointers below are never dereferenced)."""
    lib = pkv._lib
    P = ctypes.c_void_p
    good, odd = P(0x10000), P(0x10008)  # 16-byte aligned / only 8-byte aligned

    def call(out=good, q=good, Hq=32, Hkv=8, d=128, bs=16, dtype=pkv.PKV_BF16):
        return lib.pkv_paged_attention_prefill(out, q, good, good, good, 4, good, good, 2, 64, Hq, Hkv, d, bs,
                                               100, 0.1, dtype, None, None)

    assert call(Hq=30) == pkv.PKV_ERR_INVALID_ARG and b"multiple" in lib.pkv_last_error_string()
    assert call(d=64) == pkv.PKV_ERR_UNSUPPORTED
    assert call(bs=24) == pkv.PKV_ERR_UNSUPPORTED
    assert call(Hq=128) == pkv.PKV_ERR_UNSUPPORTED  # G = 16
    assert call(dtype=pkv.PKV_F32) == pkv.PKV_ERR_UNSUPPORTED
    assert call(q=odd) == pkv.PKV_ERR_UNSUPPORTED and b"aligned" in lib.pkv_last_error_string()
    assert call(out=odd) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_paged_attention_prefill(None, None, None, None, None, 4, None, None, 0, 64, 32, 8, 128, 16, 100,
                                           0.1, pkv.PKV_BF16, None, None) == pkv.PKV_OK  # empty batch


def test_quantization_compatibility_matches_the_page_and_the_oracle(pkv, orc):
    g = load_golden("quantization_cases.json")
    for c in g["cases"]:
        st = pkv._lib.pkv_validate_quantization_compatibility(g["scheme_tags"][c["scheme"]], c["axis"],
                                                              c["block_size"], g["page_size"])
        assert (st == pkv.PKV_OK) == c["valid"], c["note"]
    for tag in range(0, 6):
        for axis in range(0, 4):
            for bsz in (1, 4, 8, 16):
                for ps in (4, 16):
                    st = pkv._lib.pkv_validate_quantization_compatibility(tag, axis, bsz, ps)
                    assert (st == pkv.PKV_OK) == (orc.quantization_compatible(tag, axis, bsz, ps) == 0)
    pkv.pkv_validate_quantization_compatibility(pkv.QUANT_PER_BLOCK, 0, 16, 16)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_validate_quantization_compatibility(pkv.QUANT_PER_BLOCK, 0, 8, 16)
    assert pkv._lib.pkv_validate_quantization_compatibility(3, 0, 4, 0) == pkv.PKV_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_code8_argument_errors_are_synchronous(pkv, fmt):
    """The 8-bit cache entries (E4M3 and int8) reject bad sizes, NULL pointers
    and fp32 queries before any CUDA call, and treat empty work as a no-op."""
    lib = pkv._lib
    quant = getattr(lib, "pkv_quantize_kvcache_" + fmt)
    store = getattr(lib, "pkv_store_kvcache_" + fmt)
    attend = getattr(lib, "pkv_paged_attention_decode_" + fmt)
    assert quant(None, None, None, 4, 16, 8, 127, pkv.PKV_BF16, None) == pkv.PKV_ERR_INVALID_ARG  # odd head_dim
    assert b"even" in lib.pkv_last_error_string() and fmt.encode() in lib.pkv_last_error_string()
    assert quant(None, None, None, 4, 16, 8, 128, 9, None) == pkv.PKV_ERR_INVALID_ARG  # unknown dtype
    assert quant(None, None, None, 4, 16, 8, 128, pkv.PKV_BF16, None) == pkv.PKV_ERR_INVALID_ARG  # NULL
    assert quant(None, None, None, 0, 16, 8, 128, pkv.PKV_BF16, None) == pkv.PKV_OK  # no blocks
    assert store(None, None, None, None, None, None, None, 3, 8, 128, 64, 16, pkv.PKV_BF16, None, None) == \
        pkv.PKV_ERR_INVALID_ARG
    assert store(None, None, None, None, None, None, None, 0, 8, 128, 64, 16, pkv.PKV_BF16, None, None) == pkv.PKV_OK
    args = (None, None, None, None, None, None, None, 4, None, 2, 16, 8, 128, 16, 10, 64, 0.1)
    assert attend(*args, pkv.PKV_BF16, None, 0, None, None) == pkv.PKV_ERR_INVALID_ARG  # NULL scales
    assert b"scales" in lib.pkv_last_error_string()
    P = ctypes.c_void_p(0x10000)
    args = (None, None, None, None, P, P, None, 4, None, 2, 16, 8, 128, 16, 10, 64, 0.1)
    assert attend(*args, pkv.PKV_F32, None, 0, None, None) == pkv.PKV_ERR_UNSUPPORTED
    args = (None, None, None, None, None, None, None, 4, None, 0, 16, 8, 128, 16, 10, 64, 0.1)
    assert attend(*args, pkv.PKV_BF16, None, 0, None, None) == pkv.PKV_OK  # empty batch


def test_selftest_wait_timeout_argument_errors_are_synchronous(pkv):
    """The failure-detection self-test refuses a missing flag and limits outside
    (0, 1 s] before any launch."""
    lib = pkv._lib
    P = ctypes.c_void_p(0x10000)
    assert lib.pkv_selftest_wait_timeout(None, 1000, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(ctypes.c_void_p(0x10002), 1000, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(P, 0, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_selftest_wait_timeout(P, 1000001, None) == pkv.PKV_ERR_INVALID_ARG
    assert b"timeout" in lib.pkv_last_error_string()
