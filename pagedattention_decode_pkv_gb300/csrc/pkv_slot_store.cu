// Slot mapping and the slot-mapping scatter (store_kvcache).
//
// "Paged KV Cache - AI infra interview lesson":
//   - "Walk the Shapes First": the slot of position p is
//     block_table[p // bs] * bs + p % bs, and slot_mapping covers only the
//     tokens computed in this step.
//   - "Step 1: slot_mapping and store_kvcache": the cache is addressed as
//     [num_blocks * bs, H_kv * d] rows; row slot receives the token's K (and
//     V); slot -1 is padding and is not written.
//
// Both kernels are HBM/latency bound.  The scatter moves each row with 16-byte
// vectors: one warp owns a (token, 2 KiB segment) work item, every lane keeps
// four K and four V vectors in flight before storing them.
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "pkv_pdl.cuh"

namespace pkv {
namespace {

constexpr int kSlotThreads = 256;

// One CTA per sequence; threads stride over the sequence's new positions.
__global__ void __launch_bounds__(kSlotThreads)
slot_mapping_kernel(const int32_t *__restrict__ block_tables, int32_t max_blocks,
                    const int32_t *__restrict__ starts, const int32_t *__restrict__ ends,
                    const int32_t *__restrict__ cu_new, int32_t block_size, int32_t num_blocks,
                    int32_t *__restrict__ slot_mapping, int64_t num_new_tokens,
                    int32_t *__restrict__ err_flag) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int32_t start = starts[b], end = ends[b];
    const int64_t out0 = cu_new[b], out1 = cu_new[b + 1];
    int64_t count = static_cast<int64_t>(end) - start;
    if (count < 0) count = 0;
    int64_t writable = count;
    if (out1 - out0 != count || out0 < 0 || out0 + count > num_new_tokens) {
        // cu_new disagrees with [start, end): write only what fits the span.
        if (threadIdx.x == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_SPAN);
        int64_t span = out1 - out0;
        if (out0 < 0) span = 0;
        if (out0 + span > num_new_tokens) span = num_new_tokens - out0;
        writable = span < count ? span : count;
        if (writable < 0) writable = 0;
    }
    const int32_t *row = block_tables + static_cast<int64_t>(b) * max_blocks;
    bool bad = false;
    for (int64_t k = threadIdx.x; k < writable; k += blockDim.x) {
        const int64_t p = start + k;
        const int64_t logical = p / block_size;
        int32_t slot = -1;
        if (p >= 0 && logical < max_blocks) {
            const int32_t phys = row[logical];
            if (phys >= 0 && phys < num_blocks)
                slot = static_cast<int32_t>(static_cast<int64_t>(phys) * block_size + p % block_size);
        }
        bad |= (slot < 0);
        slot_mapping[out0 + k] = slot;
    }
    if (bad && err_flag) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
}

template <int VEC>
struct VecType;
template <> struct VecType<16> { using T = int4; };
template <> struct VecType<8> { using T = int2; };
template <> struct VecType<4> { using T = int; };
template <> struct VecType<2> { using T = short; };

constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 4;

// Work item = (token i, segment of 32 * kStoreUnroll vectors of its row).
template <int VEC>
__global__ void __launch_bounds__(kStoreThreads)
store_kvcache_kernel(const char *__restrict__ key, const char *__restrict__ value,
                     char *__restrict__ k_cache, char *__restrict__ v_cache,
                     const int32_t *__restrict__ slot_mapping, int64_t num_tokens,
                     int64_t row_bytes, int64_t num_slots, int32_t *__restrict__ err_flag) {
    pdl_wait();
    pdl_trigger();
    using V = typename VecType<VEC>::T;
    constexpr int64_t kSeg = 32LL * kStoreUnroll * VEC;
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (kStoreThreads / 32);
    const int64_t nseg = (row_bytes + kSeg - 1) / kSeg;
    const int64_t items = num_tokens * nseg;
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * (kStoreThreads / 32) + (threadIdx.x >> 5);
         item < items; item += warps_total) {
        const int64_t i = item / nseg;
        const int64_t seg = item - i * nseg;
        const int32_t slot = __ldg(slot_mapping + i);
        if (slot == -1) continue;  // padding: not written
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0 && seg == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_SLOT_RANGE);
            continue;
        }
        const int64_t src = i * row_bytes + seg * kSeg;
        const int64_t dst = static_cast<int64_t>(slot) * row_bytes + seg * kSeg;
        V kv[kStoreUnroll], vv[kStoreUnroll];
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t off = (static_cast<int64_t>(u) * 32 + lane) * VEC;
            if (seg * kSeg + off < row_bytes) {
                kv[u] = __ldcs(reinterpret_cast<const V *>(key + src + off));
                vv[u] = __ldcs(reinterpret_cast<const V *>(value + src + off));
            }
        }
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t off = (static_cast<int64_t>(u) * 32 + lane) * VEC;
            if (seg * kSeg + off < row_bytes) {
                *reinterpret_cast<V *>(k_cache + dst + off) = kv[u];
                *reinterpret_cast<V *>(v_cache + dst + off) = vv[u];
            }
        }
    }
}

int sm_count() {
    static int count = [] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        return n;
    }();
    return count;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_compute_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                               const int32_t *starts, const int32_t *ends,
                                               const int32_t *cu_new, int32_t num_seqs,
                                               int32_t block_size, int32_t num_blocks,
                                               int32_t *slot_mapping, int64_t num_new_tokens,
                                               int32_t *err_flag, void *stream) {
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || num_blocks < 0 ||
        num_new_tokens < 0)
        return set_error(PKV_ERR_INVALID_ARG,
                         "slot mapping: bad sizes (num_seqs=%d max_blocks=%d block_size=%d "
                         "num_blocks=%d num_new_tokens=%lld)",
                         num_seqs, max_blocks_per_seq, block_size, num_blocks,
                         (long long)num_new_tokens);
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return set_error(PKV_ERR_INVALID_ARG, "slot mapping: num_blocks * block_size >= 2^31");
    if (num_seqs == 0) return ok();
    if (!starts || !ends || !cu_new || (max_blocks_per_seq > 0 && !block_tables) ||
        (num_new_tokens > 0 && !slot_mapping))
        return set_error(PKV_ERR_INVALID_ARG, "slot mapping: NULL pointer");
    cudaError_t e = launch_pdl(kPdlSlotMapping, slot_mapping_kernel, dim3(num_seqs), dim3(kSlotThreads), 0,
                               static_cast<cudaStream_t>(stream), block_tables, max_blocks_per_seq, starts, ends,
                               cu_new, block_size, num_blocks, slot_mapping, num_new_tokens, err_flag);
    if (e != cudaSuccess)
        return set_error(PKV_ERR_CUDA, "slot mapping launch: %s", cudaGetErrorString(e));
    return ok();
}

extern "C" pkv_status pkv_store_kvcache(const void *key, const void *value, void *k_cache,
                                        void *v_cache, const int32_t *slot_mapping,
                                        int64_t num_tokens, int32_t num_kv_heads,
                                        int32_t head_dim, int64_t num_slots, pkv_dtype dtype,
                                        int32_t *err_flag, void *stream) {
    const int64_t es = dtype_bytes(dtype);
    if (es == 0) return set_error(PKV_ERR_INVALID_ARG, "store: unknown dtype %d", (int)dtype);
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_slots < 0)
        return set_error(PKV_ERR_INVALID_ARG, "store: bad sizes");
    if (num_tokens == 0) return ok();
    if (!key || !value || !k_cache || !v_cache || !slot_mapping)
        return set_error(PKV_ERR_INVALID_ARG, "store: NULL pointer");
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * es;
    // widest vector that divides the row and every base address
    int vec = 16;
    while (vec > es && (row_bytes % vec || !aligned(key, vec) || !aligned(value, vec) ||
                        !aligned(k_cache, vec) || !aligned(v_cache, vec)))
        vec >>= 1;
    if (row_bytes % vec || !aligned(key, vec) || !aligned(value, vec) || !aligned(k_cache, vec) ||
        !aligned(v_cache, vec))
        return set_error(PKV_ERR_INVALID_ARG, "store: buffers not aligned to the element size");
    const int64_t seg = 32LL * kStoreUnroll * vec;
    const int64_t items = num_tokens * ((row_bytes + seg - 1) / seg);
    const int64_t warps_per_cta = kStoreThreads / 32;
    int64_t grid = (items + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    if (grid > cap) grid = cap;
    auto s = static_cast<cudaStream_t>(stream);
    auto kc = static_cast<char *>(k_cache);
    auto vc = static_cast<char *>(v_cache);
    auto kk = static_cast<const char *>(key);
    auto vv = static_cast<const char *>(value);
    cudaError_t e;
    switch (vec) {
    case 16: e = launch_pdl(kPdlStore, store_kvcache_kernel<16>, dim3(grid), dim3(kStoreThreads), 0, s, kk, vv, kc, vc, slot_mapping, num_tokens, row_bytes, num_slots, err_flag); break;
    case 8: e = launch_pdl(kPdlStore, store_kvcache_kernel<8>, dim3(grid), dim3(kStoreThreads), 0, s, kk, vv, kc, vc, slot_mapping, num_tokens, row_bytes, num_slots, err_flag); break;
    case 4: e = launch_pdl(kPdlStore, store_kvcache_kernel<4>, dim3(grid), dim3(kStoreThreads), 0, s, kk, vv, kc, vc, slot_mapping, num_tokens, row_bytes, num_slots, err_flag); break;
    default: e = launch_pdl(kPdlStore, store_kvcache_kernel<2>, dim3(grid), dim3(kStoreThreads), 0, s, kk, vv, kc, vc, slot_mapping, num_tokens, row_bytes, num_slots, err_flag); break;
    }
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "store launch: %s", cudaGetErrorString(e));
    return ok();
}
