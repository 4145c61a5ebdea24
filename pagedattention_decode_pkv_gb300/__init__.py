"""Paged-KV hot path for GB300 (sm_103a): thin Python binding of libpkv.so.

Every function here has the name of the C entry point it calls (declared in
include/pkv.h) and only marshals arguments: it checks tensor placement, dtype
and shape, allocates outputs with torch, and passes raw pointers plus the
current CUDA stream.  All computation happens in the library's CUDA kernels;
if libpkv.so has not been built, importing this package fails.

Sources: "Paged KV Cache - AI infra interview lesson" (Walk the Shapes First;
Step 1: slot_mapping and store_kvcache; Step 2: paged_attention_decode) and
"Block-Paged KV Cache" (The three buffers; Element lookup through the block
table; Validating the storage invariants).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libpkv.so")

if not os.path.exists(LIBRARY_PATH):
    raise ImportError(
        f"{LIBRARY_PATH} is not built; run `python pagedattention_decode_pkv_gb300/build.py` "
        "(nvcc, sm_103a) first")

_lib = ctypes.CDLL(LIBRARY_PATH)

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_OUT_OF_RANGE, \
    PKV_ERR_WORKSPACE = range(6)
PKV_F32, PKV_F16, PKV_BF16 = 0, 1, 2
PKV_U32, PKV_U64 = 0, 1
ERRBIT_SLOT_RANGE, ERRBIT_BLOCK_RANGE, ERRBIT_CONTEXT, ERRBIT_CSR_PAGE, ERRBIT_CSR_PHYS, \
    ERRBIT_SPAN, ERRBIT_TIMEOUT = 0x01, 0x02, 0x04, 0x08, 0x10, 0x20, 0x40
_DTYPE = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}

_vp, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "pkv_last_error_string": ([], ctypes.c_char_p),
    "pkv_version": ([], ctypes.c_char_p),
    "pkv_compute_slot_mapping": ([_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i64, _vp, _vp], ctypes.c_int),
    "pkv_store_kvcache": ([_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, ctypes.c_int, _vp, _vp], ctypes.c_int),
    "pkv_paged_attention_decode": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                    _f32, ctypes.c_int, _vp, _sz, _vp, _vp], ctypes.c_int),
    "pkv_paged_attention_decode_append": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                           _i32, _i32, _i32, _f32, ctypes.c_int, _vp, _sz, _vp, _vp], ctypes.c_int),
    "pkv_paged_attention_decode_static_ws": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                              _i32, _i32, _f32, ctypes.c_int, _vp, _vp], ctypes.c_int),
    "pkv_paged_attention_decode_workspace_size": ([_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int], _sz),
    "pkv_paged_attention_decode_plan": ([_i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _vp, _vp, _vp],
                                        ctypes.c_int),
    "pkv_unpack_block_paged": ([_vp, _vp, _vp, _vp, ctypes.c_int, _vp, _i32, _i64, _i32, _i64, _i32, _i32, _i64,
                                ctypes.c_int, _vp, _vp], ctypes.c_int),
    "pkv_validate_index_buffers": ([_vp, _vp, ctypes.c_int, _i64, _i64, _i64], ctypes.c_int),
    "pkv_validate_quantization_compatibility": ([_i32, _i32, _i32, _i32], ctypes.c_int),
    "pkv_validate_token_ptr": ([_vp, _vp, ctypes.c_int, _i64, _i32, _i64], ctypes.c_int),
    "pkv_validate_block_paged_shape": ([_vp, _i32, _i32, _i32], ctypes.c_int),
    "pkv_block_paged_element_offset": ([_i64, _i64, _i64, _i64, _i32, _i64, _i32, _i32, _vp, _vp, ctypes.c_int,
                                        _i64, _vp], ctypes.c_int),
    "pkv_paged_attention_prefill": ([_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                     _i32, _f32, ctypes.c_int, _vp, _vp], ctypes.c_int),
    "pkv_quantize_kvcache_fp8": ([_vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_int, _vp], ctypes.c_int),
    "pkv_store_kvcache_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, _i32, ctypes.c_int, _vp,
                               _vp], ctypes.c_int),
    "pkv_paged_attention_decode_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                        _i32, _i32, _f32, ctypes.c_int, _vp, _sz, _vp, _vp], ctypes.c_int),
    "pkv_quantize_kvcache_int8": ([_vp, _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_int, _vp], ctypes.c_int),
    "pkv_store_kvcache_int8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, _i32, ctypes.c_int, _vp,
                                _vp], ctypes.c_int),
    "pkv_paged_attention_decode_int8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                         _i32, _i32, _f32, ctypes.c_int, _vp, _sz, _vp, _vp], ctypes.c_int),
    "pkv_paged_attention_decode_append_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                               _i32, _i32, _i32, _i32, _i32, _f32, ctypes.c_int, _vp, _sz, _vp, _vp],
                                              ctypes.c_int),
    "pkv_paged_attention_decode_append_int8": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                                _i32, _i32, _i32, _i32, _i32, _f32, ctypes.c_int, _vp, _sz, _vp, _vp],
                                               ctypes.c_int),
    "pkv_selftest_wait_timeout": ([_vp, ctypes.c_uint32, _vp], ctypes.c_int),
    "pkv_allocator_create": ([_i32, _i32, _vp], ctypes.c_int),
    "pkv_allocator_destroy": ([_vp], None),
    "pkv_allocator_add_sequence": ([_vp, _i64, _i64, _vp], ctypes.c_int),
    "pkv_allocator_fork": ([_vp, _i64, _i64, _i64], ctypes.c_int),
    "pkv_allocator_append": ([_vp, _i64, _i64, _vp], ctypes.c_int),
    "pkv_allocator_release": ([_vp, _i64], ctypes.c_int),
    "pkv_allocator_block_table": ([_vp, _i64, _vp, _i32, _vp, _vp], ctypes.c_int),
    "pkv_allocator_stats": ([_vp, _vp, _vp, _vp, _vp], ctypes.c_int),
    "pkv_allocator_check": ([_vp], _i32),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status}: {message}")
        self.status = status


def _check(status: int):
    if status != PKV_OK:
        raise PkvError(status, _lib.pkv_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*tensors):
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one CUDA device, got {devs}")
    d = devs.pop()
    if d.type != "cuda":
        raise ValueError("tensors must be CUDA tensors (no CPU path exists)")
    for t in tensors:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    return d


def _stream(dev, stream):
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return ctypes.c_void_p(s.cuda_stream)


def _want(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def pkv_version() -> str:
    return _lib.pkv_version().decode()


def pkv_compute_slot_mapping(block_tables, starts, ends, cu_new, block_size: int, num_blocks: int, *,
                             num_new_tokens: int | None = None, out=None, err_flag=None, stream=None):
    """int32 slot of every position in [starts[b], ends[b]) of every sequence, at cu_new[b]..."""
    dev = _dev(block_tables, starts, ends, cu_new, out, err_flag)
    for t, n in ((block_tables, "block_tables"), (starts, "starts"), (ends, "ends"), (cu_new, "cu_new")):
        _want(t, torch.int32, n)
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    B = block_tables.shape[0]
    if starts.numel() != B or ends.numel() != B or cu_new.numel() != B + 1:
        raise ValueError("starts/ends need num_seqs entries and cu_new num_seqs+1")
    if out is None:
        if num_new_tokens is None:
            num_new_tokens = int(cu_new[-1].item()) if B else 0  # host read: pass num_new_tokens to avoid it
        out = torch.empty(num_new_tokens, dtype=torch.int32, device=dev)
    _want(out, torch.int32, "out")
    with torch.cuda.device(dev):
        _check(_lib.pkv_compute_slot_mapping(_ptr(block_tables), block_tables.shape[1], _ptr(starts), _ptr(ends),
                                             _ptr(cu_new), B, block_size, num_blocks, _ptr(out), out.numel(),
                                             _ptr(err_flag), _stream(dev, stream)))
    return out


def pkv_store_kvcache(key, value, k_cache, v_cache, slot_mapping, *, err_flag=None, stream=None):
    """In place: k_cache/v_cache rows slot_mapping[i] <- key[i]/value[i]; slot -1 skipped."""
    dev = _dev(key, value, k_cache, v_cache, slot_mapping, err_flag)
    _want(slot_mapping, torch.int32, "slot_mapping")
    if key.dtype not in _DTYPE or not (key.dtype == value.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("key, value and caches must share one of float32/float16/bfloat16")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_blocks, block_size, num_kv_heads, head_dim]")
    nb, bs, H, d = k_cache.shape
    N = slot_mapping.numel()
    if key.shape != (N, H, d) or value.shape != (N, H, d):
        raise ValueError(f"key/value must be [{N}, {H}, {d}]")
    with torch.cuda.device(dev):
        _check(_lib.pkv_store_kvcache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), N,
                                      H, d, nb * bs, _DTYPE[key.dtype], _ptr(err_flag), _stream(dev, stream)))


def pkv_paged_attention_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                              max_context_len, dtype) -> int:
    return int(_lib.pkv_paged_attention_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                              block_size, max_context_len, _DTYPE[dtype]))


def pkv_paged_attention_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_context_len, dtype):
    """(tokens per partition, number of partitions, fast path used)."""
    p, n, f = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.pkv_paged_attention_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                                max_context_len, _DTYPE[dtype], ctypes.byref(p), ctypes.byref(n),
                                                ctypes.byref(f)))
    return p.value, n.value, bool(f.value)


def pkv_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                               max_context_len: int, *, out=None, workspace=None, err_flag=None, stream=None):
    """out[b, h] = softmax(scale * q[b, h] . K^T) V over the sequence's paged context."""
    return _decode(q, None, None, k_cache, v_cache, block_tables, context_lens, scale, max_context_len, out,
                   workspace, err_flag, stream)


def pkv_paged_attention_decode_append(q, key, value, k_cache, v_cache, block_tables, context_lens, scale: float,
                                      max_context_len: int, *, out=None, workspace=None, err_flag=None,
                                      stream=None):
    """One decode step: key[b] / value[b] go to the cache row of position
    context_lens[b] - 1, then the attention of pkv_paged_attention_decode runs
    over the whole context (new token included)."""
    return _decode(q, key, value, k_cache, v_cache, block_tables, context_lens, scale, max_context_len, out,
                   workspace, err_flag, stream)


def _decode(q, key, value, k_cache, v_cache, block_tables, context_lens, scale, max_context_len, out, workspace,
            err_flag, stream):
    dev = _dev(q, key, value, k_cache, v_cache, block_tables, context_lens, out, workspace, err_flag)
    if (key is None) != (value is None):
        raise ValueError("key and value go together")
    if key is not None:
        if key.dtype != q.dtype or value.dtype != q.dtype or key.shape != value.shape or \
                key.shape != (q.shape[0], k_cache.shape[2], q.shape[2]) or not key.is_contiguous() or \
                not value.is_contiguous():
            raise ValueError("key, value: contiguous [num_seqs, num_kv_heads, head_dim] of the cache dtype")
    _want(block_tables, torch.int32, "block_tables")
    _want(context_lens, torch.int32, "context_lens")
    if q.dtype not in _DTYPE or not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q and caches must share one of float32/float16/bfloat16")
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape or block_tables.dim() != 2:
        raise ValueError("q [B, Hq, d], caches [num_blocks, bs, Hkv, d], block_tables [B, max_blocks]")
    B, Hq, d = q.shape
    nb, bs, Hkv, d2 = k_cache.shape
    if d2 != d or context_lens.numel() != B or block_tables.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    ws = pkv_paged_attention_decode_workspace_size(B, Hq, Hkv, d, bs, max_context_len, q.dtype) if B else 0
    if ws and workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    wsp = _ptr(workspace) if ws else None
    wsn = workspace.numel() * workspace.element_size() if ws else 0
    with torch.cuda.device(dev):
        if key is None:
            _check(_lib.pkv_paged_attention_decode(
                _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                _ptr(context_lens), B, Hq, Hkv, d, bs, nb, max_context_len, float(scale), _DTYPE[q.dtype],
                wsp, wsn, _ptr(err_flag), _stream(dev, stream)))
        else:
            _check(_lib.pkv_paged_attention_decode_append(
                _ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, d, bs, nb, max_context_len, float(scale),
                _DTYPE[q.dtype], wsp, wsn, _ptr(err_flag), _stream(dev, stream)))
    return out


_INDEX = {torch.int32: PKV_U32, torch.uint32: PKV_U32, torch.int64: PKV_U64, torch.uint64: PKV_U64}


def pkv_unpack_block_paged(page_pool, block_table, seq_ptr, token_ptr, *, total_tokens: int | None = None,
                           out=None, err_flag=None, stream=None):
    """Contiguous [total_tokens, num_heads, head_dim] of one {kv_role, layer} snapshot."""
    dev = _dev(page_pool, block_table, seq_ptr, token_ptr, out, err_flag)
    if block_table.dtype != seq_ptr.dtype or block_table.dtype not in _INDEX:
        raise TypeError("block_table and seq_ptr must share a 32- or 64-bit integer type")
    _want(token_ptr, torch.int64, "token_ptr")
    if page_pool.dim() != 4 or page_pool.dtype not in _DTYPE:
        raise ValueError("page_pool must be [num_pages, page_size, num_heads, head_dim] float32/16/bf16")
    num_pages, ps, H, d = page_pool.shape
    S = seq_ptr.numel() - 1
    if token_ptr.numel() != S + 1:
        raise ValueError("token_ptr needs num_seqs + 1 entries")
    if out is None:
        if total_tokens is None:
            total_tokens = int(token_ptr[-1].item())  # host read: pass total_tokens to avoid it
        out = torch.empty(total_tokens, H, d, dtype=page_pool.dtype, device=dev)
    shape = (ctypes.c_int64 * out.dim())(*out.shape)
    _check(_lib.pkv_validate_block_paged_shape(shape, out.dim(), H, d))
    with torch.cuda.device(dev):
        _check(_lib.pkv_unpack_block_paged(_ptr(out), _ptr(page_pool), _ptr(block_table), _ptr(seq_ptr),
                                           _INDEX[block_table.dtype], _ptr(token_ptr), S, block_table.numel(), ps,
                                           num_pages, H, d, out.shape[0], _DTYPE[page_pool.dtype], _ptr(err_flag),
                                           _stream(dev, stream)))
    return out


def _host_index(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    elif t.dtype not in _INDEX:
        t = t.to(torch.int64)
    return t.cpu().contiguous()


def pkv_validate_index_buffers(seq_ptr, block_table, num_pages: int, index_dtype=None):
    """Raises PkvError unless the page's four storage invariants hold (host data)."""
    sp = _host_index(seq_ptr, index_dtype)
    bt = _host_index(block_table, sp.dtype)
    _check(_lib.pkv_validate_index_buffers(_ptr(sp), _ptr(bt) if bt.numel() else None, _INDEX[sp.dtype],
                                           sp.numel() - 1, bt.numel(), num_pages))


QUANT_NONE, QUANT_PER_TENSOR, QUANT_PER_CHANNEL, QUANT_PER_BLOCK = 0x00, 0x01, 0x02, 0x03


def pkv_validate_quantization_compatibility(scheme_tag: int, axis: int, block_size: int, page_size: int):
    """Raises PkvError unless the scheme's scales fit the block-paged layout:
    per-block-affine along the paged axis (0) with block_size == page_size;
    per-channel not along the paged axis."""
    _check(_lib.pkv_validate_quantization_compatibility(scheme_tag, axis, block_size, page_size))


def pkv_validate_token_ptr(token_ptr, seq_ptr, page_size: int, total_tokens: int, index_dtype=None):
    tp = _host_index(token_ptr, torch.int64)
    sp = _host_index(seq_ptr, index_dtype)
    _check(_lib.pkv_validate_token_ptr(_ptr(tp), _ptr(sp), _INDEX[sp.dtype], sp.numel() - 1, page_size,
                                       total_tokens))


def pkv_validate_block_paged_shape(shape, num_heads: int, head_dim: int):
    arr = (ctypes.c_int64 * max(1, len(shape)))(*shape)
    _check(_lib.pkv_validate_block_paged_shape(arr, len(shape), num_heads, head_dim))


def pkv_block_paged_element_offset(seq, token, head, dim, page_size, num_pages, num_heads, head_dim,
                                   block_table, seq_ptr, index_dtype=None) -> int:
    sp = _host_index(seq_ptr, index_dtype)
    bt = _host_index(block_table, sp.dtype)
    flat = ctypes.c_int64()
    _check(_lib.pkv_block_paged_element_offset(seq, token, head, dim, page_size, num_pages, num_heads, head_dim,
                                               _ptr(bt), _ptr(sp), _INDEX[sp.dtype], sp.numel() - 1,
                                               ctypes.byref(flat)))
    return flat.value


def pkv_paged_attention_prefill(q, k_cache, v_cache, block_tables, starts, cu_q, scale: float, max_q_len: int, *,
                                out=None, err_flag=None, stream=None):
    """Causal prefill: query i of sequence b (row cu_q[b] + i of q, position
    starts[b] + i) attends over positions 0 .. starts[b] + i of its paged context."""
    dev = _dev(q, k_cache, v_cache, block_tables, starts, cu_q, out, err_flag)
    _want(block_tables, torch.int32, "block_tables")
    _want(starts, torch.int32, "starts")
    _want(cu_q, torch.int32, "cu_q")
    if q.dtype not in _DTYPE or not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q and caches must share one of float32/float16/bfloat16")
    Tq, Hq, d = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    B = starts.numel()
    if cu_q.numel() != B + 1 or block_tables.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    with torch.cuda.device(dev):
        _check(_lib.pkv_paged_attention_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                                block_tables.shape[1], _ptr(starts), _ptr(cu_q), B, max_q_len, Hq,
                                                Hkv, d, bs, nb, float(scale), _DTYPE[q.dtype], _ptr(err_flag),
                                                _stream(dev, stream)))
    return out


# ----------------------------------------------------------------------------- 8-bit (E4M3 / int8) caches
# Code caches: E4M3 as torch.uint8 bytes, int8 as torch.int8.
_CODES = {"fp8": torch.uint8, "int8": torch.int8}


def _quantize_codes(fmt, cache, codes, scales, stream):
    dev = _dev(cache, codes, scales)
    if cache.dtype not in _DTYPE or cache.dim() != 4:
        raise ValueError("cache: [num_blocks, bs, Hkv, d] of float32/float16/bfloat16")
    nb, bs, H, d = cache.shape
    if codes is None:
        codes = torch.empty(cache.shape, dtype=_CODES[fmt], device=dev)
    if scales is None:
        scales = torch.empty(nb, H, dtype=torch.float32, device=dev)
    _want(codes, _CODES[fmt], "codes")
    _want(scales, torch.float32, "scales")
    fn = getattr(_lib, "pkv_quantize_kvcache_" + fmt)
    with torch.cuda.device(dev):
        _check(fn(_ptr(cache), _ptr(codes), _ptr(scales), nb, bs, H, d, _DTYPE[cache.dtype], _stream(dev, stream)))
    return codes, scales


def _store_codes(fmt, key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, err_flag, stream):
    dev = _dev(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, err_flag)
    _want(slot_mapping, torch.int32, "slot_mapping")
    _want(k_cache, _CODES[fmt], "k_cache")
    _want(v_cache, _CODES[fmt], "v_cache")
    nb, bs, H, d = k_cache.shape
    fn = getattr(_lib, "pkv_store_kvcache_" + fmt)
    with torch.cuda.device(dev):
        _check(fn(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                  _ptr(slot_mapping), slot_mapping.numel(), H, d, nb * bs, bs, _DTYPE[key.dtype], _ptr(err_flag),
                  _stream(dev, stream)))


def _attention_codes(fmt, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                     max_context_len, out, workspace, err_flag, stream, key=None, value=None):
    dev = _dev(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out, workspace, err_flag, key,
               value)
    _want(k_cache, _CODES[fmt], "k_cache")
    _want(v_cache, _CODES[fmt], "v_cache")
    _want(k_scale, torch.float32, "k_scale")
    _want(v_scale, torch.float32, "v_scale")
    _want(block_tables, torch.int32, "block_tables")
    _want(context_lens, torch.int32, "context_lens")
    B, Hq, d = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    ws = pkv_paged_attention_decode_workspace_size(B, Hq, Hkv, d, bs, max_context_len, q.dtype) if B else 0
    if ws and workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    tail = (block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, d, bs, nb, max_context_len, float(scale),
            _DTYPE[q.dtype], _ptr(workspace) if ws else None,
            workspace.numel() * workspace.element_size() if ws else 0, _ptr(err_flag), _stream(dev, stream))
    with torch.cuda.device(dev):
        if key is None:
            fn = getattr(_lib, "pkv_paged_attention_decode_" + fmt)
            _check(fn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                      _ptr(block_tables), *tail))
        else:
            if key.dtype != q.dtype or value.dtype != q.dtype or key.shape != (B, Hkv, d) or value.shape != key.shape:
                raise ValueError("key/value must be [num_seqs, num_kv_heads, head_dim] of the q dtype")
            fn = getattr(_lib, "pkv_paged_attention_decode_append_" + fmt)
            _check(fn(_ptr(out), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache),
                      _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), *tail))
    return out


def pkv_quantize_kvcache_fp8(cache, *, codes=None, scales=None, stream=None):
    """[num_blocks, bs, Hkv, d] cache -> (uint8 E4M3 codes of the same shape,
    float32 scales [num_blocks, Hkv]); per (block, head) s = max|x| / 448."""
    return _quantize_codes("fp8", cache, codes, scales, stream)


def pkv_store_kvcache_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, *, err_flag=None,
                          stream=None):
    """Writes encode(key[i] / s) into row slot_mapping[i] of the E4M3 code caches (in place)."""
    _store_codes("fp8", key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, err_flag, stream)


def pkv_paged_attention_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                   scale: float, max_context_len: int, *, out=None, workspace=None, err_flag=None,
                                   stream=None):
    """Decode attention over E4M3 code caches with per-(block, head) scales."""
    return _attention_codes("fp8", q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                            max_context_len, out, workspace, err_flag, stream)


def pkv_paged_attention_decode_append_fp8(q, key, value, k_cache, v_cache, k_scale, v_scale, block_tables,
                                          context_lens, scale: float, max_context_len: int, *, out=None,
                                          workspace=None, err_flag=None, stream=None):
    """One decode step over E4M3 code caches: key[b] / value[b] are encoded
    under the existing (block, head) scales into the row of position
    context_lens[b] - 1 (in place), then the attention of
    pkv_paged_attention_decode_fp8 runs over the whole context."""
    return _attention_codes("fp8", q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                            max_context_len, out, workspace, err_flag, stream, key, value)


def pkv_quantize_kvcache_int8(cache, *, codes=None, scales=None, stream=None):
    """[num_blocks, bs, Hkv, d] cache -> (int8 codes of the same shape, float32
    scales [num_blocks, Hkv]); per (block, head) s = max|x| / 127."""
    return _quantize_codes("int8", cache, codes, scales, stream)


def pkv_store_kvcache_int8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, *, err_flag=None,
                           stream=None):
    """Writes encode(key[i] / s) into row slot_mapping[i] of the int8 code caches (in place)."""
    _store_codes("int8", key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, err_flag, stream)


def pkv_paged_attention_decode_int8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                    scale: float, max_context_len: int, *, out=None, workspace=None, err_flag=None,
                                    stream=None):
    """Decode attention over int8 code caches with per-(block, head) scales."""
    return _attention_codes("int8", q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                            max_context_len, out, workspace, err_flag, stream)


def pkv_paged_attention_decode_append_int8(q, key, value, k_cache, v_cache, k_scale, v_scale, block_tables,
                                           context_lens, scale: float, max_context_len: int, *, out=None,
                                           workspace=None, err_flag=None, stream=None):
    """One decode step over int8 code caches (see pkv_paged_attention_decode_append_fp8)."""
    return _attention_codes("int8", q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale,
                            max_context_len, out, workspace, err_flag, stream, key, value)


# ----------------------------------------------------------------------------- failure detection
def pkv_selftest_wait_timeout(err_flag, timeout_us: int, *, stream=None):
    """Runs the bounded pipeline wait on a barrier nothing completes: after
    `timeout_us` the kernel sets ERRBIT_TIMEOUT in `err_flag` (device int32)."""
    dev = _dev(err_flag)
    _want(err_flag, torch.int32, "err_flag")
    with torch.cuda.device(dev):
        _check(_lib.pkv_selftest_wait_timeout(_ptr(err_flag), int(timeout_us), _stream(dev, stream)))


# ----------------------------------------------------------------------------- host block allocator
class BlockAllocator:
    """Handle of a host block allocator (see pkv_allocator_* in pkv.h); the
    pool is freed with the object."""

    def __init__(self, num_blocks: int, block_size: int):
        h = ctypes.c_void_p()
        _check(_lib.pkv_allocator_create(num_blocks, block_size, ctypes.byref(h)))
        self._h, self.num_blocks, self.block_size = h, num_blocks, block_size

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            _lib.pkv_allocator_destroy(h)


def pkv_allocator_create(num_blocks: int, block_size: int) -> BlockAllocator:
    return BlockAllocator(num_blocks, block_size)


def pkv_allocator_add_sequence(a: BlockAllocator, seq: int, num_tokens: int, blocks=None):
    arr = None
    if blocks is not None:
        blocks = list(blocks)
        arr = (ctypes.c_int32 * max(1, len(blocks)))(*blocks)
        if len(blocks) < -(-num_tokens // a.block_size):
            raise ValueError("blocks must cover num_tokens")
    _check(_lib.pkv_allocator_add_sequence(a._h, seq, num_tokens, arr))


def pkv_allocator_fork(a: BlockAllocator, parent: int, child: int, num_tokens: int):
    _check(_lib.pkv_allocator_fork(a._h, parent, child, num_tokens))


def pkv_allocator_append(a: BlockAllocator, seq: int, num_tokens: int = 1) -> list:
    """Grows the sequence; returns the slots of its new positions."""
    arr = (ctypes.c_int32 * max(1, num_tokens))()
    _check(_lib.pkv_allocator_append(a._h, seq, num_tokens, arr))
    return list(arr[:num_tokens])


def pkv_allocator_release(a: BlockAllocator, seq: int):
    _check(_lib.pkv_allocator_release(a._h, seq))


def pkv_allocator_block_table(a: BlockAllocator, seq: int, max_blocks: int):
    """(row of max_blocks block ids padded with -1, length in tokens, blocks used)."""
    row = (ctypes.c_int32 * max(1, max_blocks))()
    n, used = ctypes.c_int64(), ctypes.c_int32()
    _check(_lib.pkv_allocator_block_table(a._h, seq, row, max_blocks, ctypes.byref(n), ctypes.byref(used)))
    return list(row[:max_blocks]), n.value, used.value


def pkv_allocator_stats(a: BlockAllocator) -> dict:
    v = [ctypes.c_int64() for _ in range(4)]
    _check(_lib.pkv_allocator_stats(a._h, *[ctypes.byref(x) for x in v]))
    return dict(zip(("free", "allocated", "referenced", "sequences"), (x.value for x in v)))


def pkv_allocator_check(a: BlockAllocator) -> int:
    return int(_lib.pkv_allocator_check(a._h))
