"""CPU oracle for the paged-KV hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product library
(``pagedattention_decode_pkv_gb300``) never imports it, and the two share no
code: the arithmetic lives in ``pkv_oracle.c`` (plain per-element loops in
binary64), and this module only marshals CPU tensors into it with ctypes.

Sources are cited per function in ``pkv_oracle.c``:
"Block-Paged KV Cache" (Hurray format documentation) and
"Paged KV Cache - AI infra interview lesson".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_SO = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into libpkv_oracle.so next to it (plain C, gcc)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, u64, dbl, vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.orc_widen_f16.argtypes = [ctypes.c_uint16]
            lib.orc_widen_f16.restype = dbl
            lib.orc_widen_bf16.argtypes = [ctypes.c_uint16]
            lib.orc_widen_bf16.restype = dbl
            lib.orc_slot_of_position.argtypes = [vp, i32, i64, i32]
            lib.orc_slot_of_position.restype = i64
            lib.orc_compute_slot_mapping.argtypes = [vp, i32, vp, vp, i32, i32, i32, vp]
            lib.orc_compute_slot_mapping.restype = i64
            lib.orc_store_kvcache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64]
            lib.orc_store_kvcache.restype = i64
            lib.orc_paged_attention_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                       i32, i32, i32, i32, dbl, ctypes.c_int]
            lib.orc_paged_attention_decode.restype = i64
            lib.orc_validate_index_buffers.argtypes = [vp, vp, ctypes.c_int, i64, i64, u64]
            lib.orc_validate_index_buffers.restype = ctypes.c_int
            lib.orc_quantization_compatible.argtypes = [ctypes.c_int] * 4
            lib.orc_quantization_compatible.restype = ctypes.c_int
            lib.orc_element_offset.argtypes = [i64, i64, i64, i64, i64, u64, i64, i64, vp, vp,
                                               ctypes.c_int, i64]
            lib.orc_element_offset.restype = i64
            lib.orc_unpack_block_paged.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, i64, i64,
                                                   u64, i64, i64, i64]
            lib.orc_unpack_block_paged.restype = i64
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = dbl
            lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_int8_encode.argtypes = [ctypes.c_float]
            lib.orc_int8_encode.restype = ctypes.c_int8
            lib.orc_quantize_kvcache_q8.argtypes = [vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int]
            lib.orc_quantize_kvcache_q8.restype = None
            lib.orc_store_kvcache_q8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                 ctypes.c_int, ctypes.c_int]
            lib.orc_store_kvcache_q8.restype = i64
            lib.orc_paged_attention_decode_q8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                          i32, i32, i32, i32, dbl, ctypes.c_int, ctypes.c_int]
            lib.orc_paged_attention_decode_q8.restype = i64
            lib.orc_paged_attention_prefill.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                                        i32, i32, dbl, ctypes.c_int]
            lib.orc_paged_attention_prefill.restype = i64
            _lib = lib
    return _lib


def _cpu(t: torch.Tensor, dtype=None) -> torch.Tensor:
    t = t.detach()
    if dtype is not None:
        t = t.to(dtype)
    return t.cpu().contiguous()


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def widen_f16(bits: int) -> float:
    return _load().orc_widen_f16(bits)


def widen_bf16(bits: int) -> float:
    return _load().orc_widen_bf16(bits)


def slot_of_position(block_table_row, p: int, block_size: int) -> int:
    row = _cpu(torch.as_tensor(block_table_row), torch.int32)
    return _load().orc_slot_of_position(_ptr(row), row.numel(), p, block_size)


def compute_slot_mapping(block_tables, starts, ends, block_size: int, num_blocks: int):
    """Returns (slot_mapping int32 [sum(end-start)], error count)."""
    bt = _cpu(torch.as_tensor(block_tables), torch.int32)
    if bt.dim() == 1:
        bt = bt[None]
    st = _cpu(torch.as_tensor(starts), torch.int32).reshape(-1)
    en = _cpu(torch.as_tensor(ends), torch.int32).reshape(-1)
    total = int((en - st).clamp(min=0).sum())
    out = torch.empty(total, dtype=torch.int32)
    err = _load().orc_compute_slot_mapping(_ptr(bt), bt.shape[1], _ptr(st), _ptr(en),
                                           st.numel(), block_size, num_blocks, _ptr(out))
    return out, err


def store_kvcache(key, value, k_cache, v_cache, slot_mapping):
    """In-place on CPU copies of the caches; returns (k_cache, v_cache, error count)."""
    key, value = _cpu(key), _cpu(value)
    kc, vc = _cpu(k_cache).clone(), _cpu(v_cache).clone()
    sm = _cpu(slot_mapping, torch.int32)
    n = sm.numel()
    row_bytes = key[0].numel() * key.element_size() if n else 0
    num_slots = kc.shape[0] * kc.shape[1]
    err = _load().orc_store_kvcache(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc), _ptr(sm), n,
                                    row_bytes, num_slots)
    return kc, vc, err


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float):
    """Binary64 output [B, Hq, d] and error count.  q and caches share one dtype."""
    q, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    assert q.dtype == kc.dtype == vc.dtype
    bt = _cpu(block_tables, torch.int32)
    cl = _cpu(context_lens, torch.int32)
    B, Hq, d = q.shape
    nb, bs, Hkv, d2 = kc.shape
    assert d2 == d and Hq % Hkv == 0
    out = torch.empty(B, Hq, d, dtype=torch.float64)
    err = _load().orc_paged_attention_decode(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                             bt.shape[1] if bt.dim() == 2 else 0, _ptr(cl), B, Hq,
                                             Hkv, d, bs, nb, float(scale), _DTYPE_CODE[q.dtype])
    return out, err


def decode_step(q, key, value, k_cache, v_cache, block_tables, context_lens, scale: float):
    """One decode step as the walk in "Walk the Shapes First" runs it: the new
    token of sequence b sits at position context_lens[b] - 1, its slot comes
    from compute_slot_mapping over [ctx - 1, ctx), store_kvcache writes key[b]
    and value[b] there, and paged_attention_decode attends over the whole
    context.  Sequences with an empty context append nothing.  Returns
    (binary64 output, k_cache, v_cache, error count) with CPU copies of the
    caches."""
    cl = _cpu(context_lens, torch.int32)
    keep = (cl > 0).nonzero().reshape(-1)
    bt = _cpu(block_tables, torch.int32)
    nb = _cpu(k_cache).shape[0]
    slots, e1 = compute_slot_mapping(bt[keep], cl[keep] - 1, cl[keep], _cpu(k_cache).shape[1], nb)
    kc, vc, e2 = store_kvcache(_cpu(key)[keep], _cpu(value)[keep], k_cache, v_cache, slots)
    out, e3 = paged_attention_decode(q, kc, vc, bt, cl, scale)
    return out, kc, vc, e1 + e2 + e3


def e4m3_decode(code: int) -> float:
    """Value of an 8-bit E4M3 code (OCP FP8)."""
    return _load().orc_e4m3_decode(code)


def e4m3_encode(x: float) -> int:
    """binary32 -> E4M3 code: round to nearest even, saturating at +-448."""
    return int(_load().orc_e4m3_encode(x))


_Q8 = {"fp8": (0, torch.uint8), "int8": (1, torch.int8)}  # code format, code dtype


def _quantize_q8(cache, fmt):
    code, cdt = _Q8[fmt]
    src = _cpu(cache)
    nb, bs, H, d = src.shape
    codes = torch.empty(nb, bs, H, d, dtype=cdt)
    scales = torch.empty(nb, H, dtype=torch.float32)
    _load().orc_quantize_kvcache_q8(_ptr(src), _ptr(codes), _ptr(scales), nb, bs, H, d, _DTYPE_CODE[src.dtype],
                                    code)
    return codes, scales


def _store_q8(key, value, k_codes, v_codes, k_scale, v_scale, slot_mapping, fmt):
    code, cdt = _Q8[fmt]
    key, value = _cpu(key), _cpu(value)
    kc, vc = _cpu(k_codes).clone(), _cpu(v_codes).clone()
    assert kc.dtype == cdt and vc.dtype == cdt
    ks, vs = _cpu(k_scale, torch.float32), _cpu(v_scale, torch.float32)
    sm = _cpu(slot_mapping, torch.int32)
    nb, bs, H, d = kc.shape
    err = _load().orc_store_kvcache_q8(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(sm),
                                       sm.numel(), H, d, bs, nb * bs, _DTYPE_CODE[key.dtype], code)
    return kc, vc, err


def _attention_q8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale, fmt):
    code, cdt = _Q8[fmt]
    q = _cpu(q)
    kc, vc = _cpu(k_codes), _cpu(v_codes)
    ks, vs = _cpu(k_scale, torch.float32), _cpu(v_scale, torch.float32)
    bt = _cpu(block_tables, torch.int32)
    cl = _cpu(context_lens, torch.int32)
    B, Hq, d = q.shape
    nb, bs, Hkv, d2 = kc.shape
    assert d2 == d and Hq % Hkv == 0 and kc.dtype == cdt and vc.dtype == cdt
    out = torch.empty(B, Hq, d, dtype=torch.float64)
    err = _load().orc_paged_attention_decode_q8(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                                _ptr(bt), bt.shape[1] if bt.dim() == 2 else 0, _ptr(cl), B, Hq,
                                                Hkv, d, bs, nb, float(scale), _DTYPE_CODE[q.dtype], code)
    return out, err


def quantize_kvcache_fp8(cache):
    """[num_blocks, bs, H, d] cache -> (uint8 E4M3 codes of the same shape,
    float32 scales [num_blocks, H]); per (block, head) s = max|x| / 448."""
    return _quantize_q8(cache, "fp8")


def store_kvcache_fp8(key, value, k_codes, v_codes, k_scale, v_scale, slot_mapping):
    """fp8 "Step 1" on CPU copies of the code caches; returns (k_codes,
    v_codes, error count)."""
    return _store_q8(key, value, k_codes, v_codes, k_scale, v_scale, slot_mapping, "fp8")


def paged_attention_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale: float):
    """Binary64 output [B, Hq, d] and error count over an fp8 cache."""
    return _attention_q8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale, "fp8")


def int8_encode(x: float) -> int:
    """binary32 -> int8 code: round to nearest even, clamp to [-127, 127], NaN -> 0."""
    return int(_load().orc_int8_encode(x))


def quantize_kvcache_int8(cache):
    """[num_blocks, bs, H, d] cache -> (int8 codes of the same shape, float32
    scales [num_blocks, H]); per (block, head) s = max|x| / 127."""
    return _quantize_q8(cache, "int8")


def store_kvcache_int8(key, value, k_codes, v_codes, k_scale, v_scale, slot_mapping):
    """int8 "Step 1" on CPU copies of the code caches; returns (k_codes,
    v_codes, error count)."""
    return _store_q8(key, value, k_codes, v_codes, k_scale, v_scale, slot_mapping, "int8")


def paged_attention_decode_int8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale: float):
    """Binary64 output [B, Hq, d] and error count over an int8 cache."""
    return _attention_q8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale, "int8")


def paged_attention_prefill(q, k_cache, v_cache, block_tables, starts, cu_q, scale: float):
    """Causal prefill attention over the paged cache: q [cu_q[-1], Hq, d], the
    queries of sequence b at positions starts[b] + i.  Binary64 output of q's
    shape and the error count."""
    q, kc, vc = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    assert q.dtype == kc.dtype == vc.dtype
    bt = _cpu(block_tables, torch.int32)
    st = _cpu(starts, torch.int32).reshape(-1)
    cu = _cpu(cu_q, torch.int32).reshape(-1)
    Tq, Hq, d = q.shape
    nb, bs, Hkv, d2 = kc.shape
    assert d2 == d and Hq % Hkv == 0 and cu.numel() == st.numel() + 1
    out = torch.empty(Tq, Hq, d, dtype=torch.float64)
    err = _load().orc_paged_attention_prefill(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                              bt.shape[1] if bt.dim() == 2 else 0, _ptr(st), _ptr(cu), st.numel(),
                                              Hq, Hkv, d, bs, nb, float(scale), _DTYPE_CODE[q.dtype])
    return out, err


def validate_index_buffers(seq_ptr, block_table, num_pages: int, index_dtype=torch.int64) -> int:
    """0 when p1's four storage invariants hold, else the first broken one (1..4)."""
    is_u64 = index_dtype in (torch.int64, torch.uint64)
    tdt = torch.int64 if is_u64 else torch.int32
    sp = _cpu(torch.as_tensor(seq_ptr), tdt)
    bt = _cpu(torch.as_tensor(block_table), tdt)
    return _load().orc_validate_index_buffers(_ptr(sp), _ptr(bt), int(is_u64), sp.numel() - 1,
                                              bt.numel(), num_pages)


def quantization_compatible(scheme_tag: int, axis: int, block_size: int, page_size: int) -> int:
    """0 when the quantization scheme fits the block-paged layout, else the
    broken rule (1..4, see orc_quantization_compatible)."""
    return _load().orc_quantization_compatible(scheme_tag, axis, block_size, page_size)


def element_offset(seq, token, head, dim, page_size, num_pages, num_heads, head_dim,
                   block_table, seq_ptr, index_dtype=torch.int64) -> int:
    is_u64 = index_dtype in (torch.int64, torch.uint64)
    tdt = torch.int64 if is_u64 else torch.int32
    sp = _cpu(torch.as_tensor(seq_ptr), tdt)
    bt = _cpu(torch.as_tensor(block_table), tdt)
    return _load().orc_element_offset(seq, token, head, dim, page_size, num_pages, num_heads,
                                      head_dim, _ptr(bt), _ptr(sp), int(is_u64), sp.numel() - 1)


def unpack_block_paged(page_pool, block_table, seq_ptr, token_ptr, index_dtype=torch.int64):
    """[total_tokens, H, d] in the pool's dtype, and the error count."""
    pool = _cpu(page_pool)
    num_pages, page_size, H, d = pool.shape
    is_u64 = index_dtype in (torch.int64, torch.uint64)
    tdt = torch.int64 if is_u64 else torch.int32
    sp = _cpu(torch.as_tensor(seq_ptr), tdt)
    bt = _cpu(torch.as_tensor(block_table), tdt)
    tp = _cpu(torch.as_tensor(token_ptr), torch.int64)
    total = int(tp[-1])
    out = torch.empty(total, H, d, dtype=pool.dtype)
    err = _load().orc_unpack_block_paged(_ptr(out), _ptr(pool), _ptr(bt), _ptr(sp), int(is_u64),
                                         _ptr(tp), sp.numel() - 1, page_size, num_pages, H, d,
                                         pool.element_size())
    return out, err
