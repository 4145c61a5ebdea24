// Shared-memory pipeline and tensor-core helpers of the attention kernels
// (inline PTX: mbarrier, TMA bulk tensor copies, ldmatrix, mma.sync, format
// conversions) and the host-side tensor maps over the paged pools.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kFastHeadDim = 128;  // head_dim of the tensor-core paths
constexpr int kStageTokens = 16;   // tokens per pipeline stage (one m16 MMA tile)

// ----------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Raise the transaction count the current phase waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: false once the CTA's deadline has passed without the phase
// completing.  A stage normally lands within microseconds, so the deadline
// only matters if the pipeline is broken; it keeps such a CTA from hanging.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t deadline) {
    if (mbar_try_wait(bar, parity)) return true;
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() > deadline) return false;
    }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// The same load with an L2 eviction-priority policy (createpolicy) attached.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                                 uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Fetch a tensor map (a __grid_constant__ kernel parameter) into the TMA
// unit's descriptor cache ahead of its first bulk copy.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy for data read exactly once: its lines are the first to be evicted.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 -> two f16 (round to nearest even; the 8-bit cache paths run their MMAs in f16).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Four E4M3 codes (one 32-bit word, lowest byte first) -> two f16x2 words
// holding codes (0, 1) and (2, 3), exactly (every E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// (b0, b1, b2, b3) -> (b0, b2, b1, b3): the low half pairs bytes 0 and 2, the
// high half bytes 1 and 3.
__device__ __forceinline__ uint32_t byte_pairs(uint32_t w) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(d) : "r"(w));
    return d;
}

// Code formats of the caches the decode kernel reads.
enum CacheCode { kCode16 = 0, kCodeE4M3 = 1, kCodeInt8 = 2 };

// Four int8 codes -> two f16x2 words, exactly.  Each byte, offset by 128 to an
// unsigned u (xor of its sign bit), becomes the low mantissa byte of the f16
// 1024 (0x6400 | u is 1024 + u), and 1152 = 1024 + 128 is subtracted.  The
// byte selectors SLO / SHI place the bytes: 0x4140 / 0x4342 for (0, 1) and
// (2, 3), 0x4240 / 0x4341 for (0, 2) and (1, 3).
template <uint32_t SLO, uint32_t SHI>
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    asm("prmt.b32 %0, %1, 0x64646464, %2;" : "=r"(lo) : "r"(u), "n"(SLO));
    asm("prmt.b32 %0, %1, 0x64646464, %2;" : "=r"(hi) : "r"(u), "n"(SHI));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// Four 8-bit codes of format FMT -> two f16x2 words holding codes (0, 1) and
// (2, 3), or (0, 2) and (1, 3) when PAIRS.
template <int FMT, bool PAIRS>
__device__ __forceinline__ void codes4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    if constexpr (FMT == kCodeInt8) {
        if constexpr (PAIRS) {
            s8x4_to_f16x4<0x4240u, 0x4341u>(w, lo, hi);
        } else {
            s8x4_to_f16x4<0x4140u, 0x4342u>(w, lo, hi);
        }
    } else {
        e4m3x4_to_f16x4(PAIRS ? byte_pairs(w) : w, lo, hi);
    }
}

template <typename T> struct Half16;
template <> struct Half16<__nv_bfloat16> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
        return d;
    }
    __device__ __forceinline__ static void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <> struct Half16<__half> {
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        uint32_t d;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
        return d;
    }
    __device__ __forceinline__ static void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
};

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Pool [num_slots, Hkv, 128] viewed as (64 elements, num_slots, 2*Hkv half-rows);
// a box is box_rows slots of box_halves consecutive half-rows.
pkv_status make_kv_map_box(CUtensorMap *map, const void *pool, CUtensorMapDataType type, int64_t num_slots,
                           int Hkv, int box_rows, int box_halves) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(num_slots), static_cast<cuuint64_t>(2 * Hkv)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Hkv) * kFastHeadDim * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_halves)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, type, 3, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

// The decode boxes: kStageTokens slots of hpc heads (both halves of each).
pkv_status make_kv_map(CUtensorMap *map, const void *pool, CUtensorMapDataType type, int64_t num_slots,
                       int Hkv, int hpc) {
    return make_kv_map_box(map, pool, type, num_slots, Hkv, kStageTokens, 2 * hpc);
}

}  // namespace
}  // namespace pkv
