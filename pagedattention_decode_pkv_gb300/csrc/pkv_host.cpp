// Host-side part of the library: error reporting and the CSR snapshot checks.
//
// "Block-Paged KV Cache" (Hurray format documentation):
//   - "Validating the storage invariants": seq_ptr[0] == 0, seq_ptr
//     non-decreasing, seq_ptr[num_seqs] == len(block_table), every page id
//     below num_pages; the empty batch is valid.
//   - "Element lookup through the block table": the flat page_pool offset of
//     (seq, token, head, dim).
#include <cstdio>
#include <cstring>
#include <string>

#include "pkv_internal.h"

namespace pkv {

static thread_local std::string g_last_error;

pkv_status set_error(pkv_status status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

pkv_status ok() {
    g_last_error.clear();
    return PKV_OK;
}

static inline uint64_t index_at(const void *buf, int64_t k, pkv_index_type t) {
    return t == PKV_U64 ? static_cast<const uint64_t *>(buf)[k]
                        : static_cast<uint64_t>(static_cast<const uint32_t *>(buf)[k]);
}

}  // namespace pkv

using namespace pkv;

extern "C" const char *pkv_last_error_string(void) { return g_last_error.c_str(); }

extern "C" const char *pkv_version(void) { return "pkv-gb300 0.1.0 (sm_103a)"; }

extern "C" pkv_status pkv_validate_index_buffers(const void *seq_ptr, const void *block_table,
                                                 pkv_index_type index_type, int64_t num_seqs,
                                                 int64_t nnz, int64_t num_pages) {
    if (index_type != PKV_U32 && index_type != PKV_U64)
        return set_error(PKV_ERR_INVALID_ARG, "index_type must be PKV_U32 or PKV_U64");
    if (num_seqs < 0 || nnz < 0 || num_pages < 0)
        return set_error(PKV_ERR_INVALID_ARG, "negative size (num_seqs=%lld nnz=%lld num_pages=%lld)",
                         (long long)num_seqs, (long long)nnz, (long long)num_pages);
    if (!seq_ptr || (nnz > 0 && !block_table))
        return set_error(PKV_ERR_INVALID_ARG, "NULL seq_ptr or block_table");
    if (index_at(seq_ptr, 0, index_type) != 0)
        return set_error(PKV_ERR_OUT_OF_RANGE, "seq_ptr[0] must be 0");
    for (int64_t s = 0; s < num_seqs; ++s)
        if (index_at(seq_ptr, s + 1, index_type) < index_at(seq_ptr, s, index_type))
            return set_error(PKV_ERR_OUT_OF_RANGE, "seq_ptr decreases at %lld", (long long)s);
    if (index_at(seq_ptr, num_seqs, index_type) != static_cast<uint64_t>(nnz))
        return set_error(PKV_ERR_OUT_OF_RANGE, "seq_ptr[num_seqs] != len(block_table) (%lld)",
                         (long long)nnz);
    for (int64_t k = 0; k < nnz; ++k)
        if (index_at(block_table, k, index_type) >= static_cast<uint64_t>(num_pages))
            return set_error(PKV_ERR_OUT_OF_RANGE, "block_table[%lld] >= num_pages (%lld)",
                             (long long)k, (long long)num_pages);
    return ok();
}

// "Block-Paged KV Cache", Quantization compatibility: quantization schemes
// carry over to the block-paged layout except where scales would straddle
// pages.  Per-block-affine scales must run along the paged axis (0) over
// exactly one page; per-channel scales must not run along the paged axis.
extern "C" pkv_status pkv_validate_quantization_compatibility(int32_t scheme_tag, int32_t axis,
                                                              int32_t block_size, int32_t page_size) {
    if (page_size <= 0) return set_error(PKV_ERR_INVALID_ARG, "page_size must be positive");
    switch (scheme_tag) {
    case PKV_QUANT_NONE:
    case PKV_QUANT_PER_TENSOR:
        return ok();
    case PKV_QUANT_PER_CHANNEL:
        if (axis == 0)
            return set_error(PKV_ERR_INVALID_ARG, "per-channel scales cannot run along the paged axis");
        return ok();
    case PKV_QUANT_PER_BLOCK:
        if (axis != 0)
            return set_error(PKV_ERR_INVALID_ARG, "per-block-affine scales must run along the paged axis (0), not %d",
                             (int)axis);
        if (block_size != page_size)
            return set_error(PKV_ERR_INVALID_ARG,
                             "per-block-affine block_size (%d) must equal page_size (%d): scales stay per page slot",
                             (int)block_size, (int)page_size);
        return ok();
    default:
        return set_error(PKV_ERR_INVALID_ARG, "unknown quantization scheme tag 0x%02x", (unsigned)scheme_tag);
    }
}

extern "C" pkv_status pkv_validate_token_ptr(const int64_t *token_ptr, const void *seq_ptr,
                                             pkv_index_type index_type, int64_t num_seqs,
                                             int32_t page_size, int64_t total_tokens) {
    if (index_type != PKV_U32 && index_type != PKV_U64)
        return set_error(PKV_ERR_INVALID_ARG, "index_type must be PKV_U32 or PKV_U64");
    if (!token_ptr || !seq_ptr || num_seqs < 0 || page_size <= 0 || total_tokens < 0)
        return set_error(PKV_ERR_INVALID_ARG, "bad token_ptr arguments");
    if (token_ptr[0] != 0) return set_error(PKV_ERR_OUT_OF_RANGE, "token_ptr[0] must be 0");
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t len = token_ptr[s + 1] - token_ptr[s];
        if (len < 0) return set_error(PKV_ERR_OUT_OF_RANGE, "token_ptr decreases at %lld", (long long)s);
        uint64_t pages = index_at(seq_ptr, s + 1, index_type) - index_at(seq_ptr, s, index_type);
        if (static_cast<uint64_t>((len + page_size - 1) / page_size) > pages)
            return set_error(PKV_ERR_OUT_OF_RANGE,
                             "sequence %lld holds %lld tokens but only %llu pages", (long long)s,
                             (long long)len, (unsigned long long)pages);
    }
    if (token_ptr[num_seqs] != total_tokens)
        return set_error(PKV_ERR_OUT_OF_RANGE, "token_ptr[num_seqs] != total_tokens");
    return ok();
}

extern "C" pkv_status pkv_validate_block_paged_shape(const int64_t *shape, int32_t rank,
                                                     int32_t num_heads, int32_t head_dim) {
    if (rank != 3 || !shape)
        return set_error(PKV_ERR_INVALID_ARG, "block-paged is rank-3 only ([total_tokens, num_heads, "
                                              "head_dim]); got rank %d", rank);
    if (shape[0] < 0 || shape[1] != num_heads || shape[2] != head_dim)
        return set_error(PKV_ERR_INVALID_ARG, "shape [%lld, %lld, %lld] does not match num_heads=%d head_dim=%d",
                         (long long)shape[0], (long long)shape[1], (long long)shape[2], num_heads, head_dim);
    return ok();
}

extern "C" pkv_status pkv_block_paged_element_offset(int64_t seq, int64_t token, int64_t head,
                                                     int64_t dim, int32_t page_size,
                                                     int64_t num_pages, int32_t num_heads,
                                                     int32_t head_dim, const void *block_table,
                                                     const void *seq_ptr,
                                                     pkv_index_type index_type, int64_t num_seqs,
                                                     int64_t *flat_out) {
    if (!flat_out || !seq_ptr || page_size <= 0 || num_heads <= 0 || head_dim <= 0)
        return set_error(PKV_ERR_INVALID_ARG, "bad element_offset arguments");
    if (seq < 0 || seq >= num_seqs || token < 0 || head < 0 || head >= num_heads || dim < 0 ||
        dim >= head_dim)
        return set_error(PKV_ERR_OUT_OF_RANGE, "coordinate out of range");
    const uint64_t lo = index_at(seq_ptr, seq, index_type);
    const uint64_t hi = index_at(seq_ptr, seq + 1, index_type);
    const uint64_t page_in_seq = static_cast<uint64_t>(token / page_size);
    if (lo + page_in_seq >= hi)
        return set_error(PKV_ERR_OUT_OF_RANGE, "token %lld lies beyond sequence %lld's pages",
                         (long long)token, (long long)seq);
    if (!block_table) return set_error(PKV_ERR_INVALID_ARG, "NULL block_table");
    const uint64_t phys = index_at(block_table, static_cast<int64_t>(lo + page_in_seq), index_type);
    if (phys >= static_cast<uint64_t>(num_pages))
        return set_error(PKV_ERR_OUT_OF_RANGE, "physical page %llu >= num_pages",
                         (unsigned long long)phys);
    const uint64_t row = phys * static_cast<uint64_t>(page_size) + static_cast<uint64_t>(token % page_size);
    *flat_out = static_cast<int64_t>((row * num_heads + head) * head_dim + dim);
    return ok();
}
