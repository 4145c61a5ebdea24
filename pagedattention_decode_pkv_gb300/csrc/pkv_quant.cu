// 8-bit paged caches (E4M3 fp8 or int8 codes): quantizing a 16-bit cache and
// the slot-mapping scatter into an 8-bit cache.
//
// "Block-Paged KV Cache" (Hurray format documentation), Quantization
// compatibility: per-block-affine scales with block_size == page_size stay per
// page slot, so a shared page carries its own scales.  The pages fix only that
// placement; this library keeps one binary32 scale per (physical block, KV
// head) for K and one for V ([num_blocks, Hkv]), a stored value being
// scale * decode(code).  E4M3: OCP E4M3 codes, scale = max |x| / 448; encoding
// divides by the scale in binary32 and rounds to the nearest even code,
// saturating at +-448 (cvt.rn.satfinite).  int8 (the same page names int8
// caches beside fp8 ones; symmetric reading): signed codes in [-127, 127],
// scale = max |x| / 127; encoding rounds x / scale (binary32) to the nearest
// integer, ties to even, clamps to +-127 and maps NaN to 0.  A zero scale
// stores code 0 in both formats.
//
// "Paged KV Cache - AI infra interview lesson", Step 1: slot_mapping and
// store_kvcache -- row slot of the [num_slots, Hkv * d] cache view receives the
// token's K/V; slot -1 is skipped.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "pkv_pdl.cuh"
#include "pkv_q8.cuh"

namespace pkv {
namespace {

template <typename T> __device__ __forceinline__ float widen(T x);
template <> __device__ __forceinline__ float widen<float>(float x) { return x; }
template <> __device__ __forceinline__ float widen<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float widen<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

enum CodeFormat { kE4M3 = 0, kInt8 = 1 };

// The largest code magnitude: a (block, head) scale is max |x| / this.
template <int FMT> constexpr float kCodeMax = FMT == kInt8 ? 127.f : 448.f;

// Two binary32 -> two codes (lo in the low byte) of x / s; a zero scale gives 0.
template <int FMT> __device__ __forceinline__ uint32_t encode2(float lo, float hi, float s) {
    return q8_encode2<FMT == kInt8>(lo, hi, s);
}

constexpr int kQuantThreads = 256;

// One CTA per block, one warp per head at a time: the head's bs x d values
// (bs rows of d at a stride of Hkv * d), max |x| (NaN ignored) -> s = max / kCodeMax,
// then every value -> its code.  The second pass re-reads the same bytes
// (L1/L2 resident).
template <int FMT, typename T>
__global__ void __launch_bounds__(kQuantThreads)
quantize_q8_kernel(const T *__restrict__ src, uint8_t *__restrict__ codes, float *__restrict__ scales, int32_t bs,
                    int32_t Hkv, int32_t d) {
    pdl_wait();
    pdl_trigger();
    const int64_t blk = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n2 = bs * d / 2;  // pairs of the (block, head) slice; d is even
    for (int h = warp; h < Hkv; h += kQuantThreads / 32) {
        auto at = [&](int i) -> int64_t {  // element i of (block, head): token i / d, dim i % d
            return ((blk * bs + i / d) * Hkv + h) * static_cast<int64_t>(d) + i % d;
        };
        float m = 0.f;
        for (int p = lane; p < n2; p += 32) {
            const int64_t e = at(2 * p);
            m = fmaxf(m, fmaxf(fabsf(widen(src[e])), fabsf(widen(src[e + 1]))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float s = __fdiv_rn(m, kCodeMax<FMT>);
        if (lane == 0) scales[blk * Hkv + h] = s;
        for (int p = lane; p < n2; p += 32) {
            const int64_t e = at(2 * p);
            *reinterpret_cast<uint16_t *>(codes + e) = static_cast<uint16_t>(encode2<FMT>(widen(src[e]), widen(src[e + 1]), s));
        }
    }
}

// Vector form: one warp per (block, head) slice, 16-byte loads of VEC elements;
// the slice (at most 32 * kQuantVecs vectors) stays in registers between the
// max and the encode, so the cache is read once.  Needs d % VEC == 0 and
// 16-byte aligned source rows (8-byte aligned code rows follow).
constexpr int kQuantVecs = 8;  // vectors per lane: 16 tokens x 128 dims of a 16-bit cache

template <int FMT, typename T>
__global__ void __launch_bounds__(kQuantThreads)
quantize_q8_vec_kernel(const T *__restrict__ src, uint8_t *__restrict__ codes, float *__restrict__ scales,
                        int64_t slices, int32_t bs, int32_t Hkv, int32_t d) {
    constexpr int VEC = 16 / sizeof(T);
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int vpr = d / VEC;             // vectors per token row of one head
    const int nv = bs * vpr;             // vectors per slice (<= 32 * kQuantVecs)
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32);
    for (int64_t sl = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5); sl < slices;
         sl += warps) {
        const int64_t blk = sl / Hkv;
        const int h = static_cast<int>(sl - blk * Hkv);
        uint4 v[kQuantVecs];
        int64_t off[kQuantVecs];  // element offset of each vector
#pragma unroll
        for (int k = 0; k < kQuantVecs; ++k) {
            const int i = lane + 32 * k;
            const int t = i / vpr;
            off[k] = ((blk * bs + t) * Hkv + h) * static_cast<int64_t>(d) + (i - t * vpr) * VEC;
            v[k] = i < nv ? __ldg(reinterpret_cast<const uint4 *>(src + off[k])) : make_uint4(0, 0, 0, 0);
        }
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < kQuantVecs; ++k) {
            const T *x = reinterpret_cast<const T *>(&v[k]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, fabsf(widen(x[e])));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float s = __fdiv_rn(m, kCodeMax<FMT>);
        if (lane == 0) scales[sl] = s;
#pragma unroll
        for (int k = 0; k < kQuantVecs; ++k) {
            if (lane + 32 * k >= nv) continue;
            const T *x = reinterpret_cast<const T *>(&v[k]);
            uint32_t w[VEC / 4];
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q)
                w[q] = encode2<FMT>(widen(x[4 * q]), widen(x[4 * q + 1]), s) |
                       encode2<FMT>(widen(x[4 * q + 2]), widen(x[4 * q + 3]), s) << 16;
            if constexpr (VEC == 8) {
                *reinterpret_cast<uint2 *>(codes + off[k]) = make_uint2(w[0], w[1]);
            } else {
                *reinterpret_cast<uint32_t *>(codes + off[k]) = w[0];
            }
        }
    }
}

constexpr int kStoreThreads = 256;

// One thread per (token, head, pair of dims).
template <int FMT, typename T>
__global__ void __launch_bounds__(kStoreThreads)
store_q8_kernel(const T *__restrict__ key, const T *__restrict__ value, uint8_t *__restrict__ k_codes,
                 uint8_t *__restrict__ v_codes, const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                 const int32_t *__restrict__ slot_mapping, int64_t num_tokens, int32_t Hkv, int32_t d, int32_t bs,
                 int64_t num_slots, int32_t *__restrict__ err_flag) {
    pdl_wait();
    pdl_trigger();
    const int64_t pairs_per_token = static_cast<int64_t>(Hkv) * d / 2;
    const int64_t total = num_tokens * pairs_per_token;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kStoreThreads + threadIdx.x; w < total;
         w += static_cast<int64_t>(gridDim.x) * kStoreThreads) {
        const int64_t i = w / pairs_per_token;
        const int64_t e = 2 * (w - i * pairs_per_token);  // element within the token's [Hkv, d] row
        const int32_t slot = __ldg(slot_mapping + i);
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) {
            if (e == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_SLOT_RANGE);
            continue;
        }
        const int h = static_cast<int>(e / d);
        const int64_t sidx = static_cast<int64_t>(slot / bs) * Hkv + h;
        const int64_t src = i * Hkv * static_cast<int64_t>(d) + e;
        const int64_t dst = static_cast<int64_t>(slot) * Hkv * d + e;
        const uint32_t ck = encode2<FMT>(widen(key[src]), widen(key[src + 1]), __ldg(k_scale + sidx));
        const uint32_t cv = encode2<FMT>(widen(value[src]), widen(value[src + 1]), __ldg(v_scale + sidx));
        *reinterpret_cast<uint16_t *>(k_codes + dst) = static_cast<uint16_t>(ck);
        *reinterpret_cast<uint16_t *>(v_codes + dst) = static_cast<uint16_t>(cv);
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

// Quantizes a [num_blocks, bs, Hkv, d] cache into codes + scales (`name` names
// the format in error messages).
template <int FMT>
pkv_status quantize_entry(const char *name, const void *src, void *codes, float *scales, int32_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype, void *stream) {
    if (dtype_bytes(dtype) == 0) return set_error(PKV_ERR_INVALID_ARG, "quantize %s: unknown dtype %d", name, (int)dtype);
    if (num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 2)
        return set_error(PKV_ERR_INVALID_ARG, "quantize %s: bad sizes (head_dim must be even)", name);
    if (num_blocks > INT32_MAX / 2) return set_error(PKV_ERR_INVALID_ARG, "quantize %s: too many blocks", name);
    if (num_blocks == 0) return ok();
    if (!src || !codes || !scales) return set_error(PKV_ERR_INVALID_ARG, "quantize %s: NULL pointer", name);
    if (!aligned(src, dtype_bytes(dtype)) || !aligned(codes, 2) || !aligned(scales, 4))
        return set_error(PKV_ERR_INVALID_ARG, "quantize %s: misaligned buffers", name);
    auto s = static_cast<cudaStream_t>(stream);
    auto c = static_cast<uint8_t *>(codes);
    cudaError_t e;
    const int vec = 16 / dtype_bytes(dtype);
    if (head_dim % vec == 0 && aligned(src, 16) && aligned(codes, 8) &&
        static_cast<int64_t>(block_size) * (head_dim / vec) <= 32 * kQuantVecs) {
        const int64_t slices = static_cast<int64_t>(num_blocks) * num_kv_heads;
        int64_t grid = (slices + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
        const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
        if (grid > cap) grid = cap;
        const dim3 g(static_cast<unsigned>(grid));
#define PKV_QUANT_VEC(T)                                                                                    \
    launch_pdl(kPdlStore, quantize_q8_vec_kernel<FMT, T>, g, dim3(kQuantThreads), 0, s, static_cast<const T *>(src), \
               c, scales, slices, block_size, num_kv_heads, head_dim)
        switch (dtype) {
        case PKV_BF16: e = PKV_QUANT_VEC(__nv_bfloat16); break;
        case PKV_F16: e = PKV_QUANT_VEC(__half); break;
        default: e = PKV_QUANT_VEC(float); break;
        }
#undef PKV_QUANT_VEC
        if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "quantize %s launch: %s", name, cudaGetErrorString(e));
        return ok();
    }
    const dim3 grid(static_cast<unsigned>(num_blocks));
#define PKV_QUANT(T)                                                                                              \
    launch_pdl(kPdlStore, quantize_q8_kernel<FMT, T>, grid, dim3(kQuantThreads), 0, s, static_cast<const T *>(src), c, \
               scales, block_size, num_kv_heads, head_dim)
    switch (dtype) {
    case PKV_BF16: e = PKV_QUANT(__nv_bfloat16); break;
    case PKV_F16: e = PKV_QUANT(__half); break;
    default: e = PKV_QUANT(float); break;
    }
#undef PKV_QUANT
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "quantize %s launch: %s", name, cudaGetErrorString(e));
    return ok();
}

// The slot-mapping scatter into 8-bit caches with the given scales.
template <int FMT>
pkv_status store_entry(const char *name, const void *key, const void *value, void *k_cache, void *v_cache,
                       const float *k_scale, const float *v_scale, const int32_t *slot_mapping, int64_t num_tokens,
                       int32_t num_kv_heads, int32_t head_dim, int64_t num_slots, int32_t block_size, pkv_dtype dtype,
                       int32_t *err_flag, void *stream) {
    if (dtype_bytes(dtype) == 0) return set_error(PKV_ERR_INVALID_ARG, "store %s: unknown dtype %d", name, (int)dtype);
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 2 || num_slots < 0 || block_size <= 0)
        return set_error(PKV_ERR_INVALID_ARG, "store %s: bad sizes (head_dim must be even)", name);
    if (num_tokens == 0) return ok();
    if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
        return set_error(PKV_ERR_INVALID_ARG, "store %s: NULL pointer", name);
    if (!aligned(key, dtype_bytes(dtype)) || !aligned(value, dtype_bytes(dtype)) || !aligned(k_cache, 2) ||
        !aligned(v_cache, 2) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return set_error(PKV_ERR_INVALID_ARG, "store %s: misaligned buffers", name);
    const int64_t total = num_tokens * num_kv_heads * head_dim / 2;
    int64_t grid = (total + kStoreThreads - 1) / kStoreThreads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    if (grid > cap) grid = cap;
    auto s = static_cast<cudaStream_t>(stream);
    auto kc = static_cast<uint8_t *>(k_cache);
    auto vc = static_cast<uint8_t *>(v_cache);
    cudaError_t e;
#define PKV_STORE_Q8(T)                                                                                             \
    launch_pdl(kPdlStore, store_q8_kernel<FMT, T>, dim3(static_cast<unsigned>(grid)), dim3(kStoreThreads), 0, s,    \
               static_cast<const T *>(key), static_cast<const T *>(value), kc, vc, k_scale, v_scale, slot_mapping, \
               num_tokens, num_kv_heads, head_dim, block_size, num_slots, err_flag)
    switch (dtype) {
    case PKV_BF16: e = PKV_STORE_Q8(__nv_bfloat16); break;
    case PKV_F16: e = PKV_STORE_Q8(__half); break;
    default: e = PKV_STORE_Q8(float); break;
    }
#undef PKV_STORE_Q8
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "store %s launch: %s", name, cudaGetErrorString(e));
    return ok();
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_quantize_kvcache_fp8(const void *src, void *codes, float *scales, int32_t num_blocks,
                                               int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                               pkv_dtype dtype, void *stream) {
    return quantize_entry<kE4M3>("fp8", src, codes, scales, num_blocks, block_size, num_kv_heads, head_dim, dtype,
                                 stream);
}

extern "C" pkv_status pkv_quantize_kvcache_int8(const void *src, void *codes, float *scales, int32_t num_blocks,
                                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                                pkv_dtype dtype, void *stream) {
    return quantize_entry<kInt8>("int8", src, codes, scales, num_blocks, block_size, num_kv_heads, head_dim, dtype,
                                 stream);
}

extern "C" pkv_status pkv_store_kvcache_fp8(const void *key, const void *value, void *k_cache, void *v_cache,
                                            const float *k_scale, const float *v_scale,
                                            const int32_t *slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                                            int32_t head_dim, int64_t num_slots, int32_t block_size,
                                            pkv_dtype dtype, int32_t *err_flag, void *stream) {
    return store_entry<kE4M3>("fp8", key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                              num_kv_heads, head_dim, num_slots, block_size, dtype, err_flag, stream);
}

extern "C" pkv_status pkv_store_kvcache_int8(const void *key, const void *value, void *k_cache, void *v_cache,
                                             const float *k_scale, const float *v_scale,
                                             const int32_t *slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                                             int32_t head_dim, int64_t num_slots, int32_t block_size,
                                             pkv_dtype dtype, int32_t *err_flag, void *stream) {
    return store_entry<kInt8>("int8", key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, num_tokens,
                              num_kv_heads, head_dim, num_slots, block_size, dtype, err_flag, stream);
}
