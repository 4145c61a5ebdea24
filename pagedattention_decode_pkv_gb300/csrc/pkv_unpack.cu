// CSR block-paged snapshot -> contiguous logical tensor.
//
// "Block-Paged KV Cache" (Hurray format documentation):
//   - "The three buffers": page_pool [num_pages, page_size, num_heads,
//     head_dim], block_table (physical page of every logical page, sequences
//     concatenated), seq_ptr (CSR offsets of each sequence's slice); the
//     logical shape is [total_tokens, num_heads, head_dim].
//   - "Element lookup through the block table": flat =
//     ((block_table[seq_ptr[s] + t / ps] * ps + t % ps) * H + h) * d + dim.
//
// For fixed (s, page) the formula moves whole token rows (H * d elements),
// and the rows of one page are consecutive both in the pool and in the
// output, so the gather is page-granular: every (sequence, page) pair is one
// contiguous copy of up to page_size rows.  A CTA owns pages x, x + X, ... of
// sequence blockIdx.y; threads move 16-byte vectors with eight in flight.
// Aliased pages (prefix sharing) are simply read once per referencing
// sequence; repeated reads hit L2.
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "pkv_pdl.cuh"

namespace pkv {
namespace {

constexpr int kUnpackThreads = 256;
constexpr int kUnpackUnroll = 8;

template <int VEC> struct UVec;
template <> struct UVec<16> { using T = int4; };
template <> struct UVec<8> { using T = int2; };
template <> struct UVec<4> { using T = int; };
template <> struct UVec<2> { using T = short; };

template <typename IDX, int VEC>
__global__ void __launch_bounds__(kUnpackThreads)
unpack_kernel(char *__restrict__ out, const char *__restrict__ pool,
              const IDX *__restrict__ block_table, const IDX *__restrict__ seq_ptr,
              const int64_t *__restrict__ token_ptr, int64_t nnz, int32_t page_size,
              int64_t num_pages, int64_t row_bytes, int64_t total_tokens,
              int32_t *__restrict__ err_flag) {
    pdl_wait();
    pdl_trigger();
    using V = typename UVec<VEC>::T;
    const int s = blockIdx.y;
    const uint64_t lo = seq_ptr[s], hi = seq_ptr[s + 1];
    const int64_t t0 = token_ptr[s], t1 = token_ptr[s + 1];
    if (t0 < 0 || t1 < t0 || t1 > total_tokens) {  // rows outside the output: nothing to write
        if (blockIdx.x == 0 && threadIdx.x == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_CSR_PAGE);
        return;
    }
    const int64_t len = t1 - t0;
    const int64_t pages_needed = (len + page_size - 1) / page_size;
    const bool slice_ok = lo <= hi && hi <= static_cast<uint64_t>(nnz);
    const int64_t vec_per_row = row_bytes / VEC;
    for (int64_t p = blockIdx.x; p < pages_needed; p += gridDim.x) {
        const int64_t first_row = p * page_size;
        const int64_t rows = (len - first_row) < page_size ? (len - first_row) : page_size;
        const int64_t nvec = rows * vec_per_row;
        V *dst = reinterpret_cast<V *>(out + (t0 + first_row) * row_bytes);
        int bad = 0;
        uint64_t phys = 0;
        if (!slice_ok || lo + static_cast<uint64_t>(p) >= hi) {
            bad = PKV_ERRBIT_CSR_PAGE;
        } else {
            phys = block_table[lo + p];
            if (phys >= static_cast<uint64_t>(num_pages)) bad = PKV_ERRBIT_CSR_PHYS;
        }
        if (bad) {  // unresolvable rows are zero-filled
            if (threadIdx.x == 0 && err_flag) atomicOr(err_flag, bad);
            const V zero{};
            for (int64_t v = threadIdx.x; v < nvec; v += kUnpackThreads) dst[v] = zero;
            continue;
        }
        const V *src = reinterpret_cast<const V *>(pool + static_cast<int64_t>(phys) * page_size * row_bytes);
        for (int64_t base = 0; base < nvec; base += static_cast<int64_t>(kUnpackThreads) * kUnpackUnroll) {
            V r[kUnpackUnroll];
#pragma unroll
            for (int u = 0; u < kUnpackUnroll; ++u) {
                const int64_t v = base + static_cast<int64_t>(u) * kUnpackThreads + threadIdx.x;
                if (v < nvec) r[u] = __ldg(src + v);
            }
#pragma unroll
            for (int u = 0; u < kUnpackUnroll; ++u) {
                const int64_t v = base + static_cast<int64_t>(u) * kUnpackThreads + threadIdx.x;
                if (v < nvec) __stcs(dst + v, r[u]);
            }
        }
    }
}

template <typename IDX>
cudaError_t launch_unpack(int vec, dim3 grid, cudaStream_t s, char *out, const char *pool,
                          const void *bt, const void *sp, const int64_t *tp, int64_t nnz,
                          int32_t ps, int64_t np, int64_t row_bytes, int64_t total,
                          int32_t *err) {
    auto b = static_cast<const IDX *>(bt);
    auto q = static_cast<const IDX *>(sp);
    const dim3 block(kUnpackThreads);
    switch (vec) {
    case 16: return launch_pdl(kPdlUnpack, unpack_kernel<IDX, 16>, grid, block, 0, s, out, pool, b, q, tp, nnz, ps, np, row_bytes, total, err);
    case 8: return launch_pdl(kPdlUnpack, unpack_kernel<IDX, 8>, grid, block, 0, s, out, pool, b, q, tp, nnz, ps, np, row_bytes, total, err);
    case 4: return launch_pdl(kPdlUnpack, unpack_kernel<IDX, 4>, grid, block, 0, s, out, pool, b, q, tp, nnz, ps, np, row_bytes, total, err);
    default: return launch_pdl(kPdlUnpack, unpack_kernel<IDX, 2>, grid, block, 0, s, out, pool, b, q, tp, nnz, ps, np, row_bytes, total, err);
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_unpack_block_paged(void *out, const void *page_pool, const void *block_table,
                                             const void *seq_ptr, pkv_index_type index_type,
                                             const int64_t *token_ptr, int32_t num_seqs, int64_t nnz,
                                             int32_t page_size, int64_t num_pages, int32_t num_heads,
                                             int32_t head_dim, int64_t total_tokens, pkv_dtype dtype,
                                             int32_t *err_flag, void *stream) {
    const int64_t es = dtype_bytes(dtype);
    if (es == 0) return set_error(PKV_ERR_INVALID_ARG, "unpack: unknown dtype %d", (int)dtype);
    if (index_type != PKV_U32 && index_type != PKV_U64)
        return set_error(PKV_ERR_INVALID_ARG, "unpack: index_type must be PKV_U32 or PKV_U64");
    if (num_seqs < 0 || nnz < 0 || page_size <= 0 || num_pages < 0 || num_heads <= 0 ||
        head_dim <= 0 || total_tokens < 0)
        return set_error(PKV_ERR_INVALID_ARG, "unpack: bad sizes");
    if (num_seqs > 65535)
        return set_error(PKV_ERR_UNSUPPORTED, "unpack: more than 65535 sequences in one call");
    if (num_seqs == 0 || total_tokens == 0) return ok();
    if (!out || !seq_ptr || !token_ptr || (nnz > 0 && (!block_table || !page_pool)))
        return set_error(PKV_ERR_INVALID_ARG, "unpack: NULL pointer");
    const int64_t row_bytes = static_cast<int64_t>(num_heads) * head_dim * es;
    int vec = 16;
    while (vec > es && (row_bytes % vec || !aligned(out, vec) || !aligned(page_pool, vec))) vec >>= 1;
    if (row_bytes % vec || !aligned(out, vec) || (page_pool && !aligned(page_pool, vec)))
        return set_error(PKV_ERR_INVALID_ARG, "unpack: buffers not aligned to the element size");
    // X CTAs per sequence: enough to cover the average sequence's pages in one pass.
    int64_t x = (nnz + num_seqs - 1) / num_seqs;
    if (x < 1) x = 1;
    if (x > 65535) x = 65535;
    dim3 grid(static_cast<unsigned>(x), static_cast<unsigned>(num_seqs));
    auto s = static_cast<cudaStream_t>(stream);
    cudaError_t e = index_type == PKV_U64
        ? launch_unpack<uint64_t>(vec, grid, s, static_cast<char *>(out), static_cast<const char *>(page_pool),
                                  block_table, seq_ptr, token_ptr, nnz, page_size, num_pages, row_bytes,
                                  total_tokens, err_flag)
        : launch_unpack<uint32_t>(vec, grid, s, static_cast<char *>(out), static_cast<const char *>(page_pool),
                                  block_table, seq_ptr, token_ptr, nnz, page_size, num_pages, row_bytes,
                                  total_tokens, err_flag);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "unpack launch: %s", cudaGetErrorString(e));
    return ok();
}
