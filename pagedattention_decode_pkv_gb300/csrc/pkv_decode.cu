// Paged decode attention: one query token per sequence, GQA, split-K over the
// context with a log-sum-exp combine.
//
// "Paged KV Cache - AI infra interview lesson", "Step 2: paged_attention_decode":
// n_blk = ceil(ctx / bs) block ids are taken from the sequence's table row
// (later entries may be -1); K and V are gathered through them, the unused
// tail of the last block is cut, query head h reads KV head h // (Hq / H_kv),
// and the result is softmax(q K^T * scale) V.
//
// Design (GB300, sm_103a)
// -----------------------
// The kernel is HBM-bound: every cached K/V byte of a sequence is read once.
// Work unit = (sequence b, group of HPC KV heads, partition j of the context).
// One CTA per unit runs a TMA -> shared-memory pipeline:
//   * a producer warp issues, per 16-token stage, two cp.async.bulk.tensor
//     loads (K and V) of the box [HPC heads x 2 halves x 16 tokens x 64 dims]
//     out of a 3-D tensor map over the pool viewed as
//     (64 elements, num_slots rows, 2 * H_kv half-rows), 128-byte swizzled, so
//     that the 16 tokens of one head are consecutive 128-byte rows in shared
//     memory and every ldmatrix below is bank-conflict free;
//   * one consumer warp per KV head keeps all G = Hq / H_kv query heads of its
//     group in registers (as the B operand of mma.m16n8k16, G <= 8 padded to
//     n = 8) and computes S^T = K Q^T for the 16 tokens with 8 MMAs, an online
//     softmax on the accumulator fragment (max/sum over tokens via 3 shuffles),
//     transposes P in registers with movmatrix and accumulates O^T += V^T P^T
//     with 8 more MMAs (V read with ldmatrix.trans).  Each K/V byte therefore
//     costs a handful of instructions instead of G FMAs + conversions, which
//     keeps the SMs far from the issue limit at HBM speed.
// mbarrier full/empty pairs hand stages between producer and consumers; all
// waits are bounded and report PKV_ERRBIT_TIMEOUT instead of hanging.
// A partition's output is written directly when the sequence fits in one
// partition, otherwise as an unnormalised fp32 partial (o, max, sum) that the
// combine kernel merges.  Shapes outside the fast path (fp32, other head
// dims, G > 8, block sizes not a multiple of 16) run a plain CUDA-core kernel
// with the same partitioning and the same combine.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <type_traits>

#include "pkv_internal.h"
#include "pkv_pdl.cuh"
#include "pkv_q8.cuh"
#include "pkv_tma.cuh"

namespace pkv {
namespace {

constexpr int kMaxPartition = 4096;              // tokens; bounds the per-CTA block-id list
constexpr int kMaxStagesPerPartition = kMaxPartition / kStageTokens;
constexpr int kTargetSms = 152;                  // GB300; fixed so the plan is device independent
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kCtaDeadlineNs = 2000000000ull;  // every wait of a CTA gives up 2 s after it started
constexpr int kMaxStreamSeqs = 512;    // work-balanced schedule: sequences per call (shared-memory bound)
constexpr int kMaxStreamCtas = 512;    // work-balanced schedule: CTAs per launch (sizes the workspace)
constexpr int kMinStreamStages = 4;    // work-balanced schedule: fewest stages a working CTA streams
constexpr int kChunkStages = 4;        // work-balanced schedule: dynamic-tail chunk (64 tokens)
constexpr int kTailDenominator = 6;    // work-balanced schedule: the dynamic tail is 1/6 of the stages
constexpr int kGrabAhead = 1;          // work-balanced schedule: claim the next chunk this many stages early
constexpr bool kKvEvictFirst = true;   // K/V tiles are read once: mark them first in line for L2 eviction

// ----------------------------------------------------------------------------- plan
struct Plan {
    bool fast = false;
    bool stream = false;  // fast path with the work-balanced one-wave schedule
    int groups = 1;       // work-balanced launches, one per group of <= kMaxStreamSeqs sequences
    int group_seqs = 0;   // sequences per group (the last may hold fewer)
    int64_t units = 0;    // (sequence, head group) units of the work-balanced schedule
    int64_t max_chunks = 0, max_segments = 0;  // dynamic-tail chunks / piece slots (bounds)
    size_t unit_bytes = 0;
    int hpc = 1;          // KV heads per CTA (fast path)
    int stages = 2;       // pipeline depth (fast path)
    int partition = 16;   // tokens per partition
    int nparts = 0;       // partitions covering max_context_len
    size_t o_bytes = 0;   // fp32 partial outputs
    size_t ml_bytes = 0;  // (max, sum) per partial
    size_t ws_bytes = 0;
};

int env_partition_override() {
    static int v = [] {
        const char *s = std::getenv("PKV_DECODE_PARTITION_TOKENS");
        return s ? std::atoi(s) : 0;
    }();
    return v;
}

// generic_only: plan the CUDA-core kernel (used when the fast path's pointer
// alignment does not hold at call time); max_parts > 0 caps the partitions so
// that the partials fit a workspace sized for another plan.
Plan make_plan(int B, int Hq, int Hkv, int d, int bs, int max_ctx, pkv_dtype dt, bool generic_only = false,
               int64_t max_parts = 0, bool codes8 = false) {
    Plan p;
    const int G = Hq / Hkv;
    p.fast = !generic_only && (dt == PKV_F16 || dt == PKV_BF16) && d == kFastHeadDim && G >= 1 && G <= 8 &&
             bs % kStageTokens == 0 && bs <= 32768;
    p.hpc = (Hkv % 4 == 0) ? 4 : (Hkv % 2 == 0) ? 2 : 1;
    const int stage_bytes = p.hpc * 2 * kStageTokens * kFastHeadDim * 2;
    p.stages = 98304 / stage_bytes;
    if (p.stages > 8) p.stages = 8;
    if (p.stages < 2) p.stages = 2;
    // Past kMaxStreamSeqs sequences, 16-bit caches take the fixed-partition
    // kernel (a many-wave grid: measured 7.33 TB/s on 1024 Qwen3-shaped
    // sequences); 8-bit caches, which only the work-balanced kernel reads,
    // run it as consecutive launches over groups of near-equal size that reuse
    // one scratch region in stream order (each launch's first global access
    // waits for the previous grid to complete).
    p.stream = p.fast && (B <= kMaxStreamSeqs || codes8);
    if (p.stream) {
        p.groups = B > kMaxStreamSeqs ? (B + kMaxStreamSeqs - 1) / kMaxStreamSeqs : 1;
        p.group_seqs = (B + p.groups - 1) / p.groups;
        // Pieces: at most one per (unit, segment) boundary; segments are the
        // static slices (at most kMaxStreamCtas) and the dynamic-tail chunks.
        const int64_t HG = Hkv / p.hpc, HU = Hq / HG;
        p.units = static_cast<int64_t>(p.group_seqs) * HG;
        const int64_t w_max = p.units * ((static_cast<int64_t>(max_ctx) + kStageTokens - 1) / kStageTokens);
        p.max_chunks = w_max / kTailDenominator / kChunkStages + 1;
        // static slots [0, kMaxStreamCtas + units), dynamic slots after them
        p.max_segments = 2 * p.units + kMaxStreamCtas + p.max_chunks;  // piece slots
        const size_t pieces = static_cast<size_t>(p.max_segments);
        p.o_bytes = (pieces * HU * d * sizeof(float) + 255) / 256 * 256;
        p.ml_bytes = (pieces * HU * sizeof(float2) + 255) / 256 * 256;
        p.unit_bytes = (static_cast<size_t>(p.units) * sizeof(int4) + 255) / 256 * 256;
        p.ws_bytes = p.o_bytes + p.ml_bytes + p.unit_bytes + 256;  // + Cw and the chunk counter
        p.partition = 0;
        p.nparts = 0;
        return p;
    }
    const int64_t units = static_cast<int64_t>(B) * (p.fast ? Hkv / p.hpc : Hq);
    // Aim for ~8 waves of 2 CTAs per SM; partitions are multiples of 64 tokens.
    const int64_t target = static_cast<int64_t>(kTargetSms) * 2 * 8;
    int64_t P = (static_cast<int64_t>(max_ctx) * units + target - 1) / target;
    P = ((P + 63) / 64) * 64;
    if (P < 256) P = 256;
    if (env_partition_override() > 0) P = ((env_partition_override() + 15) / 16) * 16;
    if (max_parts > 0 && (static_cast<int64_t>(max_ctx) + P - 1) / P > max_parts)
        P = ((static_cast<int64_t>(max_ctx) + max_parts - 1) / max_parts + 15) / 16 * 16;
    if (P > kMaxPartition) P = kMaxPartition;
    if (P >= max_ctx) P = ((max_ctx > 0 ? max_ctx : 1) + 15) / 16 * 16;
    if (P > kMaxPartition) P = kMaxPartition;
    p.partition = static_cast<int>(P);
    p.nparts = max_ctx > 0 ? static_cast<int>((max_ctx + P - 1) / P) : 0;
    if (p.nparts > 1) {
        const size_t rows = static_cast<size_t>(B) * Hq * p.nparts;
        p.o_bytes = (rows * d * sizeof(float) + 255) / 256 * 256;
        p.ml_bytes = (rows * sizeof(float2) + 255) / 256 * 256;
        p.ws_bytes = p.o_bytes + p.ml_bytes;
    }
    return p;
}

// Sequence-level validity shared by all kernels: a bad context length gives a
// zero row (written by partition 0) and PKV_ERRBIT_CONTEXT.
__device__ __forceinline__ bool context_ok(int ctx, int max_ctx, int bs, int max_blocks) {
    return ctx >= 0 && ctx <= max_ctx &&
           (static_cast<int64_t>(ctx) + bs - 1) / bs <= static_cast<int64_t>(max_blocks);
}

// ----------------------------------------------------------------------------- fast kernel
template <int HPC, int STAGES>
struct FastSmem {
    static constexpr int kTileBytes = HPC * 2 * kStageTokens * 128;  // one of K / V per stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kTilesBytes = STAGES * kStageBytes;
    static constexpr int kBlkOffset = kTilesBytes;
    static constexpr int kBarOffset = kBlkOffset + kMaxStagesPerPartition * 4;
    static constexpr int kFlagOffset = kBarOffset + 2 * STAGES * 8;
    static constexpr int kBytes = kFlagOffset + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

template <typename T, int HPC, int STAGES>
__global__ void __launch_bounds__((HPC + 1) * 32)
decode_fast_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   T *__restrict__ out, const T *__restrict__ q,
                   const int32_t *__restrict__ block_tables, int32_t max_blocks,
                   const int32_t *__restrict__ context_lens, int32_t Hq, int32_t G, int32_t bs,
                   int32_t num_blocks, int32_t max_ctx, int32_t partition, int32_t nparts,
                   float scale_log2, float *__restrict__ o_part, float2 *__restrict__ ml_part,
                   int32_t *__restrict__ err_flag) {
    using L = FastSmem<HPC, STAGES>;
    using H = Half16<T>;
    pdl_wait();
    pdl_trigger();
    const int j = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ctx = context_lens[b];
    const int heads_per_cta = HPC * G;
    if (!context_ok(ctx, max_ctx, bs, max_blocks) || ctx == 0) {
        if (j == 0) {
            if (ctx != 0 && threadIdx.x == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
            T *o = out + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(hg) * heads_per_cta) * kFastHeadDim;
            for (int i = threadIdx.x; i < heads_per_cta * kFastHeadDim; i += blockDim.x) o[i] = from_f32<T>(0.f);
        }
        return;
    }
    const int t0 = j * partition;
    if (t0 >= ctx) return;
    // Once any CTA has reported a broken pipeline, the rest of the launch stops early.
    if (err_flag && (*reinterpret_cast<volatile int32_t *>(err_flag) & PKV_ERRBIT_TIMEOUT)) return;
    const uint64_t deadline = global_ns() + kCtaDeadlineNs;
    const int t1 = min(t0 + partition, ctx);
    const int nstage = (t1 - t0 + kStageTokens - 1) / kStageTokens;
    const bool single = ctx <= partition;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t *sblk = reinterpret_cast<int32_t *>(smem + L::kBlkOffset);
    const uint32_t bar0 = smem_u32(smem + L::kBarOffset);  // full[s] = bar0 + 8s, empty[s] = bar0 + 8(STAGES+s)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kFlagOffset);
    const uint32_t tiles = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            mbar_init(bar0 + 8 * (STAGES + s), HPC);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == HPC) {  // producer warp: resolve this partition's block ids once
        const int32_t *row = block_tables + static_cast<int64_t>(b) * max_blocks;
        bool bad = false;
        for (int s = lane; s < nstage; s += 32) {
            const int pos = t0 + s * kStageTokens;
            int32_t id = row[pos / bs];
            if (id < 0 || id >= num_blocks) { id = -1; bad = true; }
            sblk[s] = id;
        }
        if (bad && err_flag) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
    }
    __syncthreads();

    if (warp == HPC) {
        if (lane == 0) {
            int issued = 0;
            for (int s = 0; s < nstage; ++s) {
                const int slot = s % STAGES;
                const uint32_t full = bar0 + 8 * slot, empty = bar0 + 8 * (STAGES + slot);
                if (s >= STAGES && !mbar_wait(empty, ((s / STAGES) - 1) & 1, deadline)) {
                    *abort_flag = 1;
                    if (err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
                    break;
                }
                const int id = sblk[s];
                if (id >= 0) {
                    const int slot_row = id * bs + (t0 + s * kStageTokens) % bs;
                    const uint32_t dst = tiles + slot * L::kStageBytes;
                    mbar_arrive_expect_tx(full, L::kStageBytes);
                    tma_load_3d(dst, &tm_k, 0, slot_row, 2 * hg * HPC, full);
                    tma_load_3d(dst + L::kTileBytes, &tm_v, 0, slot_row, 2 * hg * HPC, full);
                } else {
                    mbar_arrive(full);  // nothing to load: consumers mask the whole stage
                }
                issued = s + 1;
            }
            // Drain: no bulk copy may still be writing shared memory when the CTA exits.
            for (int s = issued - STAGES > 0 ? issued - STAGES : 0; s < issued; ++s)
                if (!mbar_wait(bar0 + 8 * (s % STAGES), (s / STAGES) & 1, deadline) && err_flag)
                    atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warp
    const int g = lane >> 2, t = lane & 3;
    const int hk = hg * HPC + warp;  // KV head of this warp
    uint32_t qf[8][2];
    {
        const bool live = g < G;
        const T *qrow = q + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(hk) * G + (live ? g : 0)) * kFastHeadDim;
        const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow);
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
            qf[kc][0] = live ? __ldg(q32 + kc * 8 + t) : 0u;
            qf[kc][1] = live ? __ldg(q32 + kc * 8 + 4 + t) : 0u;
        }
    }
    float o[8][4];
#pragma unroll
    for (int dc = 0; dc < 8; ++dc)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dc][e] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // Per-lane ldmatrix row offsets inside this warp's head (rows of 128 B,
    // row R = (2 * warp + half) * 16 + token, chunk swizzled with R & 7).
    const int mi = lane >> 3, r = lane & 7;
    const uint32_t head_off = static_cast<uint32_t>(warp) * 2 * kStageTokens * 128;
    uint32_t k_off[8], v_off[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        {   // QK: A = K[16 tokens x 16 dims]; matrices (tok 0-7|8-15) x (dims 0-7|8-15)
            const int tok = r + 8 * (mi & 1);
            const int c16 = 2 * c + (mi >> 1);
            const int R = ((c16 >> 3)) * kStageTokens + tok;
            k_off[c] = head_off + R * 128 + (((c16 & 7) ^ r) << 4);
        }
        {   // PV: A = V^T[16 dims x 16 tokens] via .trans; matrices (dims 0-7|8-15) x (tok 0-7|8-15)
            const int tok = r + 8 * (mi >> 1);
            const int c16 = 2 * c + (mi & 1);
            const int R = ((c16 >> 3)) * kStageTokens + tok;
            v_off[c] = head_off + R * 128 + (((c16 & 7) ^ r) << 4);
        }
    }

    for (int s = 0; s < nstage; ++s) {
        const int slot = s % STAGES;
        if (!mbar_wait(bar0 + 8 * slot, (s / STAGES) & 1, deadline) || *abort_flag) {
            if (lane == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
            return;
        }
        const uint32_t kt = tiles + slot * L::kStageBytes;
        const uint32_t vt = kt + L::kTileBytes;
        const int id = sblk[s];
        const int pos0 = t0 + s * kStageTokens;
        const int nvalid = id < 0 ? 0 : min(kStageTokens, t1 - pos0);
        if (nvalid < kStageTokens) {
            // Rows past the context (or of a skipped block) may hold anything,
            // NaN included: zero this head's V rows so 0 * row stays 0.
            const int nbad = kStageTokens - nvalid;
            for (int idx = lane; idx < nbad * 16; idx += 32) {
                const int tok = nvalid + (idx >> 4);
                const int half = (idx >> 3) & 1;
                const int chunk = idx & 7;
                const uint32_t addr = vt + head_off + (half * kStageTokens + tok) * 128 + chunk * 16;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
            }
            __syncwarp();
        }
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
            uint32_t a[4];
            ldsm_x4(kt + k_off[kc], a);
            H::mma(sc, a, qf[kc][0], qf[kc][1]);
        }
        // scores in log2 units; masked tokens -> -inf
        const bool vg = g < nvalid, vg8 = g + 8 < nvalid;
        const float x0 = vg ? sc[0] * scale_log2 : -INFINITY;
        const float x1 = vg ? sc[1] * scale_log2 : -INFINITY;
        const float x2 = vg8 ? sc[2] * scale_log2 : -INFINITY;
        const float x3 = vg8 ? sc[3] * scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float p0 = fast_exp2(x0 - base0), p1 = fast_exp2(x1 - base1);
        const float p2 = fast_exp2(x2 - base0), p3 = fast_exp2(x3 - base1);
        const float a0 = fast_exp2(m0 - base0), a1 = fast_exp2(m1 - base1);
        m0 = mn0;
        m1 = mn1;
        l0 = l0 * a0 + (p0 + p2);
        l1 = l1 * a1 + (p1 + p3);
#pragma unroll
        for (int dc = 0; dc < 8; ++dc) {
            o[dc][0] *= a0;
            o[dc][1] *= a1;
            o[dc][2] *= a0;
            o[dc][3] *= a1;
        }
        const uint32_t pb0 = movmatrix_trans(H::pack(p0, p1));
        const uint32_t pb1 = movmatrix_trans(H::pack(p2, p3));
#pragma unroll
        for (int dc = 0; dc < 8; ++dc) {
            uint32_t a[4];
            ldsm_x4_trans(vt + v_off[dc], a);
            H::mma(o[dc], a, pb0, pb1);
        }
        if (nvalid < kStageTokens) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar0 + 8 * (STAGES + slot));
    }

    // row sums over the 16 token lanes of each head column
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }
    const int hA = 2 * t, hB = 2 * t + 1;  // head columns of this lane
    const int64_t qhead0 = static_cast<int64_t>(b) * Hq + static_cast<int64_t>(hk) * G;
    if (single) {
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int dc = 0; dc < 8; ++dc) {
            const int d0 = dc * 16 + g;
            if (hA < G) {
                T *dst = out + (qhead0 + hA) * kFastHeadDim;
                dst[d0] = from_f32<T>(o[dc][0] * inv0);
                dst[d0 + 8] = from_f32<T>(o[dc][2] * inv0);
            }
            if (hB < G) {
                T *dst = out + (qhead0 + hB) * kFastHeadDim;
                dst[d0] = from_f32<T>(o[dc][1] * inv1);
                dst[d0 + 8] = from_f32<T>(o[dc][3] * inv1);
            }
        }
    } else {
#pragma unroll
        for (int dc = 0; dc < 8; ++dc) {
            const int d0 = dc * 16 + g;
            if (hA < G) {
                float *dst = o_part + ((qhead0 + hA) * nparts + j) * kFastHeadDim;
                dst[d0] = o[dc][0];
                dst[d0 + 8] = o[dc][2];
            }
            if (hB < G) {
                float *dst = o_part + ((qhead0 + hB) * nparts + j) * kFastHeadDim;
                dst[d0] = o[dc][1];
                dst[d0 + 8] = o[dc][3];
            }
        }
        if (g == 0) {
            if (hA < G) ml_part[(qhead0 + hA) * nparts + j] = make_float2(m0, l0);
            if (hB < G) ml_part[(qhead0 + hB) * nparts + j] = make_float2(m1, l1);
        }
    }
}

// ----------------------------------------------------------------------------- generic kernel
constexpr int kGenThreads = 128;

template <int NWARPS>
__device__ __forceinline__ float block_reduce_n(float v, float *scratch, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, sh);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = scratch[0];
#pragma unroll
    for (int w = 1; w < NWARPS; ++w) v = is_max ? fmaxf(v, scratch[w]) : v + scratch[w];
    return v;
}

__device__ __forceinline__ float block_reduce(float v, float *scratch, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, sh);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = scratch[0];
    for (int w = 1; w < kGenThreads / 32; ++w) v = is_max ? fmaxf(v, scratch[w]) : v + scratch[w];
    return v;
}

// One CTA per (partition, query head, sequence): scores of the partition in
// shared memory, fp32 throughout, exact exp2f.
template <typename T>
__global__ void __launch_bounds__(kGenThreads)
decode_generic_kernel(T *__restrict__ out, const T *__restrict__ q, const T *__restrict__ k_cache,
                      const T *__restrict__ v_cache, const int32_t *__restrict__ block_tables,
                      int32_t max_blocks, const int32_t *__restrict__ context_lens, int32_t Hq,
                      int32_t Hkv, int32_t d, int32_t bs, int32_t num_blocks, int32_t max_ctx,
                      int32_t partition, int32_t nparts, float scale_log2,
                      float *__restrict__ o_part, float2 *__restrict__ ml_part,
                      int32_t *__restrict__ err_flag) {
    pdl_wait();
    pdl_trigger();
    const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int ctx = context_lens[b];
    T *orow = out + (static_cast<int64_t>(b) * Hq + h) * d;
    if (!context_ok(ctx, max_ctx, bs, max_blocks) || ctx == 0) {
        if (j == 0) {
            if (ctx != 0 && threadIdx.x == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
            for (int i = threadIdx.x; i < d; i += kGenThreads) orow[i] = from_f32<T>(0.f);
        }
        return;
    }
    const int t0 = j * partition;
    if (t0 >= ctx) return;
    const int t1 = min(t0 + partition, ctx);
    const int n = t1 - t0;
    const int g = h / (Hq / Hkv);
    extern __shared__ float gsm[];
    float *qs = gsm;              // [d]
    float *sc = gsm + d;          // [partition]
    float *scratch = sc + partition;  // [32]
    const int32_t *row = block_tables + static_cast<int64_t>(b) * max_blocks;
    for (int i = threadIdx.x; i < d; i += kGenThreads) qs[i] = to_f32(q[(static_cast<int64_t>(b) * Hq + h) * d + i]);
    __syncthreads();
    bool bad = false;
    for (int k = threadIdx.x; k < n; k += kGenThreads) {
        const int pos = t0 + k;
        const int32_t id = row[pos / bs];
        if (id < 0 || id >= num_blocks) { sc[k] = -INFINITY; bad = true; continue; }
        const T *kr = k_cache + ((static_cast<int64_t>(id) * bs + pos % bs) * Hkv + g) * d;
        float acc = 0.f;
        for (int i = 0; i < d; ++i) acc = fmaf(qs[i], to_f32(kr[i]), acc);
        sc[k] = acc * scale_log2;
    }
    if (bad && err_flag) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
    float mx = -INFINITY;
    for (int k = threadIdx.x; k < n; k += kGenThreads) mx = fmaxf(mx, sc[k]);
    mx = block_reduce(mx, scratch, true);
    float lsum = 0.f;
    for (int k = threadIdx.x; k < n; k += kGenThreads) {
        const float p = mx == -INFINITY ? 0.f : exp2f(sc[k] - mx);
        sc[k] = p;
        lsum += p;
    }
    lsum = block_reduce(lsum, scratch, false);  // also orders the sc[] writes before the reads below
    for (int i = threadIdx.x; i < d; i += kGenThreads) {
        float acc = 0.f;
        for (int k = 0; k < n; ++k) {
            const float p = sc[k];
            if (p == 0.f) continue;
            const int pos = t0 + k;
            const int32_t id = row[pos / bs];
            acc = fmaf(p, to_f32(v_cache[((static_cast<int64_t>(id) * bs + pos % bs) * Hkv + g) * d + i]), acc);
        }
        if (ctx <= partition) {
            orow[i] = from_f32<T>(lsum > 0.f ? acc / lsum : 0.f);
        } else {
            o_part[((static_cast<int64_t>(b) * Hq + h) * nparts + j) * d + i] = acc;
        }
    }
    if (ctx > partition && threadIdx.x == 0)
        ml_part[(static_cast<int64_t>(b) * Hq + h) * nparts + j] = make_float2(mx, lsum);
}

// ----------------------------------------------------------------------------- combine
// out = sum_k w_k o_k / sum_k w_k,  w_k = l_k * 2^(m_k - M), M = max_k m_k (m in log2 units).
// One CTA per (query head, sequence).  The weights are computed once into
// shared memory; partitions are then spread over the four warps and the head
// dimension over the lanes (DPL dims per lane, coalesced), with four
// partitions' loads in flight per thread before they are accumulated.
constexpr int kCombineThreads = 128;
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombineUnroll = 4;

template <typename T, int DPL>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(T *__restrict__ out, const float *__restrict__ o_part, const float2 *__restrict__ ml_part,
               const int32_t *__restrict__ context_lens, int32_t Hq, int32_t d, int32_t bs,
               int32_t max_blocks, int32_t max_ctx, int32_t partition, int32_t nparts) {
    extern __shared__ float csm[];
    float *w = csm;                        // [nparts]
    float *red = csm + nparts;             // [kCombineWarps][DPL * 32]
    __shared__ float scratch[32];
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y;
    const int ctx = context_lens[b];
    if (!context_ok(ctx, max_ctx, bs, max_blocks) || ctx <= partition) return;  // written by the main kernel
    const int np = (ctx + partition - 1) / partition;
    const int64_t row = static_cast<int64_t>(b) * Hq + h;
    const float2 *ml = ml_part + row * nparts;
    float M = -INFINITY;
    for (int k = threadIdx.x; k < np; k += kCombineThreads) M = fmaxf(M, ml[k].x);
    M = block_reduce(M, scratch, true);
    float L = 0.f;
    for (int k = threadIdx.x; k < np; k += kCombineThreads) {
        const float2 v = ml[k];
        const float e = M == -INFINITY ? 0.f : exp2f(v.x - M);
        w[k] = e;
        L += v.y * e;
    }
    L = block_reduce(L, scratch, false);  // its barriers also publish w[]
    const float inv = L > 0.f ? 1.f / L : 0.f;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *base = o_part + row * nparts * static_cast<int64_t>(d);
    float acc[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
    for (int k0 = warp; k0 < np; k0 += kCombineWarps * kCombineUnroll) {
        float v[kCombineUnroll][DPL];
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
            const int k = k0 + u * kCombineWarps;
#pragma unroll
            for (int j = 0; j < DPL; ++j) {
                const int i = lane + 32 * j;
                v[u][j] = (k < np && i < d) ? __ldg(base + static_cast<int64_t>(k) * d + i) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kCombineUnroll; ++u) {
            const int k = k0 + u * kCombineWarps;
            const float wk = k < np ? w[k] : 0.f;
#pragma unroll
            for (int j = 0; j < DPL; ++j) acc[j] = fmaf(wk, v[u][j], acc[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < DPL; ++j) red[warp * DPL * 32 + lane + 32 * j] = acc[j];
    __syncthreads();
    for (int i = threadIdx.x; i < d; i += kCombineThreads) {
        float sacc = 0.f;
#pragma unroll
        for (int ww = 0; ww < kCombineWarps; ++ww) sacc += red[ww * DPL * 32 + i];
        out[row * d + i] = from_f32<T>(sacc * inv);
    }
}

template <typename T, int DPL>
cudaError_t launch_combine_dpl(T *out, const float *o_part, const float2 *ml, const int32_t *ctx, int Hq, int B,
                               int d, int bs, int max_blocks, int max_ctx, int partition, int nparts,
                               cudaStream_t s) {
    const size_t smem = (static_cast<size_t>(nparts) + kCombineWarps * DPL * 32) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(combine_kernel<T, DPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kPdlCombine, combine_kernel<T, DPL>, dim3(Hq, B), dim3(kCombineThreads), smem, s, out, o_part, ml, ctx, Hq,
                      d, bs, max_blocks, max_ctx, partition, nparts);
}

template <typename T>
cudaError_t launch_combine(T *out, const float *o_part, const float2 *ml, const int32_t *ctx, int Hq, int B, int d,
                           int bs, int max_blocks, int max_ctx, int partition, int nparts, cudaStream_t s) {
    if (d <= 32) return launch_combine_dpl<T, 1>(out, o_part, ml, ctx, Hq, B, d, bs, max_blocks, max_ctx, partition, nparts, s);
    if (d <= 64) return launch_combine_dpl<T, 2>(out, o_part, ml, ctx, Hq, B, d, bs, max_blocks, max_ctx, partition, nparts, s);
    if (d <= 128) return launch_combine_dpl<T, 4>(out, o_part, ml, ctx, Hq, B, d, bs, max_blocks, max_ctx, partition, nparts, s);
    if (d <= 256) return launch_combine_dpl<T, 8>(out, o_part, ml, ctx, Hq, B, d, bs, max_blocks, max_ctx, partition, nparts, s);
    if (d <= 512) return launch_combine_dpl<T, 16>(out, o_part, ml, ctx, Hq, B, d, bs, max_blocks, max_ctx, partition, nparts, s);
    return launch_combine_dpl<T, 32>(out, o_part, ml, ctx, Hq, B, d, bs, max_blocks, max_ctx, partition, nparts, s);
}

// ----------------------------------------------------------------------------- work-balanced kernel
// One wave of CTAs (every SM holds two).  The work of the launch is the
// flattened list of 16-token stages over (sequence b, head group hg, stage st):
// sequences in order, head groups in order, stages in order; W stages in all.
//  * Static part: every (b, hg) unit keeps about its last 1/kTailDenominator
//    (whole chunks of kChunkStages stages) as a tail; the units' other stages,
//    in order, are cut into equal contiguous slices, one per working CTA
//    ("segment" c), so every CTA moves the same number of K/V bytes whatever
//    the mix of context lengths.
//  * Dynamic tail: the units' tails, in order, form a list of chunks
//    ("segment" C + k) that CTAs claim from an atomic counter shortly before
//    they run out of work.  SMs do not all get the same share of HBM bandwidth,
//    and the chunks absorb that.
// A unit that lies wholly inside one slice and has no tail is written straight
// to `out`; otherwise every slice or chunk it touches leaves one unnormalised
// piece, at slot (c + unit) for slice c and (kMaxStreamCtas + units + k + unit)
// for chunk k, merged by stream_combine_kernel.  The producer warp describes up
// to 32 stages at a time, one batch ahead of the TMA issue (block-id loads in
// flight meanwhile), and hands each stage's (b, hg, valid rows, flags, piece
// slot) to the consumers through shared memory.
constexpr int kFlagFirst = 1 << 8;   // first stage of a piece: reset the running softmax
constexpr int kFlagLast = 1 << 9;    // last stage of a piece: flush it
constexpr int kFlagWhole = 1 << 10;  // the piece is the whole unit: write the final output
constexpr int kFlagAppend = 1 << 11; // the stage holds the step's new token: append its K/V first

// C8: the cache holds 8-bit codes (E4M3 or int8), one 128-byte row per (token,
// head), and a per-stage ring holds the (block, head) scales of K and V.
template <int HPC, int STAGES, bool C8 = false>
struct StreamSmem {
    static constexpr int kTileBytes = C8 ? HPC * kStageTokens * 128 : HPC * 2 * kStageTokens * 128;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kTilesBytes = STAGES * kStageBytes;
    static constexpr int kScaleOffset = kTilesBytes;
    static constexpr int kBatchScaleOffset = kScaleOffset + (C8 ? STAGES * 2 * HPC * 4 : 0);  // [2][32][2][HPC]
    static constexpr int kCtxOffset = kBatchScaleOffset + (C8 ? 2 * 32 * 2 * HPC * 4 : 0);  // int32 ctx per sequence
    static constexpr int kPrefOffset = kCtxOffset + 4 * kMaxStreamSeqs;   // int64 stage prefix per sequence
    static constexpr int kSPrefOffset = kPrefOffset + 8 * (kMaxStreamSeqs + 16);  // int64 static-part prefix
    static constexpr int kInfoOffset = kSPrefOffset + 8 * (kMaxStreamSeqs + 16);
    static constexpr int kBarOffset = kInfoOffset + 16 * STAGES;
    static constexpr int kFlagOffset = kBarOffset + 16 * STAGES;
    static constexpr int kBytes = kFlagOffset + 16;
    static constexpr int kAlloc = kBytes + 1024;
};

// a / b for a >= 0, b > 0.  A 64-bit division by a runtime value is a long
// dependent instruction sequence (~0.4 us for one warp on GB300), and the
// schedule below sits on the path to the first bulk copy; operands that fit
// 32 bits (always, short of ~2^31 stages) take the short unsigned form.
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t b) {
    if (((a | b) >> 32) == 0) return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
    return a / b;
}

// Tail stages of a unit with n stages: whole chunks, about n / kTailDenominator.
__device__ __forceinline__ int64_t tail_stages(int64_t n) {
    return n / kTailDenominator / kChunkStages * kChunkStages;
}

// Stage s (< HG * pre(B)) of a region whose per-sequence prefix is pre(b) ->
// sequence b, head group hg, index st inside that sequence's part.
template <typename Pre>
__device__ __forceinline__ void locate_stage(Pre pre, int B, int HG, int64_t s, int &b, int &hg, int &st) {
    int lo = 0, hi = B - 1;  // largest b with HG * pre(b) <= s (its part is not empty)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(HG) * pre(mid) <= s) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int64_t n = pre(b + 1) - pre(b);
    const int64_t off = s - static_cast<int64_t>(HG) * pre(b);
    hg = static_cast<int>(div_nonneg(off, n));
    st = static_cast<int>(off - hg * n);
}

template <typename T, int HPC, int STAGES, int FMT>
__global__ void __launch_bounds__((HPC + 1) * 32, FMT != kCode16 ? 3 : 2)
decode_stream_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     T *__restrict__ out, const T *__restrict__ q, const int32_t *__restrict__ block_tables,
                     int32_t max_blocks, const int32_t *__restrict__ context_lens, int32_t B, int32_t Hq,
                     int32_t G, int32_t HG, int32_t bs, int32_t num_blocks, int32_t max_ctx, float scale_log2,
                     float *__restrict__ o_piece, float2 *__restrict__ ml_piece, int4 *__restrict__ unit_info,
                     int32_t *__restrict__ ws_meta, uint32_t *__restrict__ chunk_ctr,
                     const T *__restrict__ new_k, const T *__restrict__ new_v, T *k_cache_w, T *v_cache_w,
                     const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                     int32_t *__restrict__ err_flag) {
    constexpr bool C8 = FMT != kCode16;  // 8-bit codes (E4M3 or int8) with per-(block, head) scales
    using L = StreamSmem<HPC, STAGES, C8>;
    using H = Half16<typename std::conditional<C8, __half, T>::type>;  // 8-bit tiles are widened to f16
    const int c = blockIdx.x, C = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t *cx = reinterpret_cast<int32_t *>(smem + L::kCtxOffset);
    int64_t *pref = reinterpret_cast<int64_t *>(smem + L::kPrefOffset);
    int64_t *spref = reinterpret_cast<int64_t *>(smem + L::kSPrefOffset);
    int4 *info = reinterpret_cast<int4 *>(smem + L::kInfoOffset);
    const uint32_t bar0 = smem_u32(smem + L::kBarOffset);  // full[s] = bar0 + 8s, empty[s] = bar0 + 8(STAGES+s)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kFlagOffset);
    const uint32_t tiles = smem_u32(smem);
    float *scl = reinterpret_cast<float *>(smem + L::kScaleOffset);  // C8: [STAGES][2][HPC] K / V scales
    float *bscl = reinterpret_cast<float *>(smem + L::kBatchScaleOffset);  // C8: [2 batches][32][2][HPC]
    auto pre_all = [&](int b) { return pref[b]; };
    auto pre_static = [&](int b) { return spref[b]; };
    auto pre_tail = [&](int b) { return pref[b] - spref[b]; };

    if (warp == HPC && lane == 0) {  // the producer's lane 0 initialises the barriers it issues on first
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar0 + 8 * i, 1);
            mbar_init(bar0 + 8 * (STAGES + i), HPC);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tm_k);  // the maps are parameters: nothing the previous grid writes
        prefetch_tensormap(&tm_v);
    }
    pdl_wait();
    pdl_trigger();
    // Chunk tickets start at 0.  Only CTA 0 resets the counter; a CTA that grabs
    // before the reset can only cause chunks to be processed twice, which writes
    // the same piece twice with identical values, and CTA 0 keeps grabbing after
    // its reset until every chunk has been handed out again.
    if (c == 0 && threadIdx.x == 0) atomicExch(chunk_ctr, 0u);
    const uint64_t deadline = global_ns() + kCtaDeadlineNs;
    // While the context lengths load, the producer guesses where its static
    // slice starts if every sequence held max_ctx tokens and loads the block ids
    // of that guess; describe() takes such an id when the real stage agrees
    // (always, for equal-length batches), which saves one dependent global
    // load before the first bulk copy.  The id is read from the same table
    // entry either way.
    int g_b = -1, g_hg = 0, g_st = 0, g_id = -1;
    const int64_t g_n = (static_cast<int64_t>(max_ctx) + kStageTokens - 1) / kStageTokens;  // stages at max_ctx
    if (warp == HPC && max_ctx > 0) {
        const int64_t n = g_n;
        const int64_t ns = n - tail_stages(n);
        const int64_t wst = static_cast<int64_t>(HG) * B * ns;
        int64_t cw = wst / kMinStreamStages;
        if (cw > C) cw = C;
        if (cw < 1) cw = 1;
        if (c < cw) {
            const int64_t sf = div_nonneg(wst * c, cw) + lane, se = div_nonneg(wst * (c + 1), cw);
            if (sf < se) {
                const int64_t unit = div_nonneg(sf, ns);
                const int st = static_cast<int>(sf - unit * ns);
                const int blk = st * kStageTokens / bs;
                if (blk < max_blocks) {
                    g_b = static_cast<int>(div_nonneg(unit, HG));
                    g_hg = static_cast<int>(unit - static_cast<int64_t>(g_b) * HG);
                    g_st = st;
                    g_id = block_tables[static_cast<int64_t>(g_b) * max_blocks + blk];
                }
            }
        }
    }
    // Early issue.  When every sequence holds max_ctx tokens the guess is the
    // real schedule, so the producer starts the bulk copies of its first stages
    // (at most STAGES, so no slot is reused) as soon as their block ids and the
    // context lengths are in, instead of after the plan and describe() below.
    // They go out under mbarrier.expect_tx alone: the stage's arrival, with its
    // info, comes when the issue loop reaches the same stage, and a slot whose
    // stage turns out different is handed to the consumers as one to skip.
    // The producer also takes the abort decision, so that a CTA with copies in
    // flight never leaves at the early return below.
    int n_early = 0;
    int e_id = -1, e_hg = 0, e_row = 0;  // lane e < n_early: stage e's block id, head group, row in block
    const uint64_t kv_policy = l2_evict_first_policy();
    if (warp == HPC) {
        int abort_now = 0;
        if (lane == 0 && err_flag)  // a broken pipeline elsewhere in the launch stops this CTA early
            abort_now = (*reinterpret_cast<volatile int32_t *>(err_flag) & PKV_ERRBIT_TIMEOUT) ? 1 : 0;
        abort_now = __shfl_sync(0xffffffffu, abort_now, 0);
        if (lane == 0) *abort_flag = abort_now;
        // (checked for up to 128 sequences: four independent loads per lane)
        bool equal = !abort_now && max_ctx > 0 && B <= 128 &&
                     g_n * kStageTokens <= static_cast<int64_t>(max_blocks) * bs;
        if (equal) {
            int lens[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) lens[k] = lane + 32 * k < B ? context_lens[lane + 32 * k] : max_ctx;
#pragma unroll
            for (int k = 0; k < 4; ++k) equal = equal && lens[k] == max_ctx;
        }
        equal = __all_sync(0xffffffffu, equal);
        if (equal) {
            const bool ok = lane < STAGES && g_b >= 0 && g_id >= 0 && g_id < num_blocks &&
                            !(new_k && g_st == g_n - 1);  // an append stage must write its row first
            n_early = __ffs(~__ballot_sync(0xffffffffu, ok)) - 1;  // the leading run of ok lanes
            if (lane < n_early) {
                const int pos0 = g_st * kStageTokens;
                e_id = g_id;
                e_hg = g_hg;
                e_row = pos0 - pos0 / bs * bs;
            }
            for (int e = 0; e < n_early; ++e) {
                const int id = __shfl_sync(0xffffffffu, e_id, e), hg = __shfl_sync(0xffffffffu, e_hg, e);
                const int row = __shfl_sync(0xffffffffu, e_row, e);
                if (lane == 0) {
                    const uint32_t full = bar0 + 8 * e, dst = tiles + e * L::kStageBytes;
                    const int z = C8 ? hg * HPC : 2 * hg * HPC;
                    mbar_expect_tx(full, L::kStageBytes);
                    if (kKvEvictFirst) {
                        tma_load_3d_hint(dst, &tm_k, 0, id * bs + row, z, full, kv_policy);
                        tma_load_3d_hint(dst + L::kTileBytes, &tm_v, 0, id * bs + row, z, full, kv_policy);
                    } else {
                        tma_load_3d(dst, &tm_k, 0, id * bs + row, z, full);
                        tma_load_3d(dst + L::kTileBytes, &tm_v, 0, id * bs + row, z, full);
                    }
                }
            }
        }
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int ctx = context_lens[b];
        cx[b] = context_ok(ctx, max_ctx, bs, max_blocks) ? ctx : 0;
    }
    __syncthreads();
    if (warp == 0) {  // exclusive prefixes of stages and of static-part stages per sequence
        const int chunk = (B + 31) / 32;
        const int lo = min(lane * chunk, B), hi = min(lo + chunk, B);
        int64_t sum = 0, ssum = 0;
        for (int b = lo; b < hi; ++b) {
            const int64_t n = (cx[b] + kStageTokens - 1) / kStageTokens;
            sum += n;
            ssum += n - tail_stages(n);
        }
        int64_t incl = sum, sincl = ssum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
            const int64_t sv = __shfl_up_sync(0xffffffffu, sincl, o);
            if (lane >= o) {
                incl += v;
                sincl += sv;
            }
        }
        int64_t run = incl - sum, srun = sincl - ssum;
        for (int b = lo; b < hi; ++b) {
            pref[b] = run;
            spref[b] = srun;
            const int64_t n = (cx[b] + kStageTokens - 1) / kStageTokens;
            run += n;
            srun += n - tail_stages(n);
        }
        if (lane == 31) {
            pref[B] = incl;
            spref[B] = sincl;
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    const int64_t W = static_cast<int64_t>(HG) * pref[B];
    const int64_t Wst = static_cast<int64_t>(HG) * spref[B];  // static region
    const int64_t K = (W - Wst) / kChunkStages;                // dynamic chunks
    const int64_t U = static_cast<int64_t>(B) * HG;
    const int64_t dyn_base = kMaxStreamCtas + U;              // first dynamic piece slot
    // Working CTAs of the static part: at most one per kMinStreamStages stages,
    // so every static slice is non-empty.
    int64_t Cw = Wst / kMinStreamStages;
    if (Cw > C) Cw = C;
    if (Cw < 1) Cw = Wst > 0 ? 1 : 0;
    const int64_t s0 = c < Cw ? div_nonneg(Wst * c, Cw) : 0, s1 = c < Cw ? div_nonneg(Wst * (c + 1), Cw) : 0;
    if (c == 0 && threadIdx.x == 0) ws_meta[0] = static_cast<int32_t>(Cw);

    // Sequences with nothing to stream (empty or invalid context) get zero rows
    // from CTA b mod C.
    for (int b = c; b < B; b += C) {
        if (cx[b] > 0) continue;
        if (threadIdx.x == 0 && context_lens[b] != 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
        T *o = out + static_cast<int64_t>(b) * Hq * kFastHeadDim;
        for (int i = threadIdx.x; i < Hq * kFastHeadDim; i += blockDim.x) o[i] = from_f32<T>(0.f);
    }
    if (W == 0) return;

    if (warp == HPC) {
        // ------------------------------------------------------------ producer warp
        // A batch = up to 32 consecutive stages [sb, se) of one segment [lo, hi).
        bool bad = false;
        // Stage sb + lane of a batch [sb, se) that lies in segment [lo, hi) of
        // the static region (seg = c) or of the dynamic region (seg = C + k).
        int cbuf = 0;  // C8: the batch-scale buffer of the current batch (the next one uses cbuf ^ 1)
        auto describe = [&](int64_t sb, int64_t se, int64_t lo, int64_t hi, int seg, int &b, int &hg,
                            int &meta, int &id, int &slot_of_piece, int buf) {
            b = hg = meta = slot_of_piece = 0;
            id = -1;
            const int64_t sf = sb + lane;
            if (sf >= se) return;
            const bool dyn = seg >= C;
            int sp;  // index inside the sequence's part
            if (dyn) locate_stage(pre_tail, B, HG, sf, b, hg, sp);
            else locate_stage(pre_static, B, HG, sf, b, hg, sp);
            const int ctx = cx[b];
            const int64_t n = pref[b + 1] - pref[b];
            const int64_t ns = spref[b + 1] - spref[b], nt = n - ns;
            const int st = dyn ? static_cast<int>(ns) + sp : sp;  // stage inside the unit
            const int pos0 = st * kStageTokens;
            const int blk = pos0 / bs, in_blk = pos0 - blk * bs;
            if (b == g_b && hg == g_hg && st == g_st) id = g_id;  // the guess was right: same table entry
            else id = block_tables[static_cast<int64_t>(b) * max_blocks + blk];  // checked when issued
            const int64_t u = static_cast<int64_t>(b) * HG + hg;
            int flags = 0;
            if (sf == lo || (!dyn && sp == 0)) flags |= kFlagFirst;
            if (sf == hi - 1 || (!dyn && sp == ns - 1)) flags |= kFlagLast;
            if (!dyn) {
                const int64_t u0 = static_cast<int64_t>(HG) * spref[b] + static_cast<int64_t>(hg) * ns;
                if (nt == 0 && u0 >= lo && u0 + ns <= hi) flags |= kFlagWhole;
                slot_of_piece = static_cast<int>(seg + u);
                if (sp == 0) unit_info[u].x = seg;
                if (sp == ns - 1) {  // the unit's static part ends here: record its chunk range too
                    const int64_t t0 = static_cast<int64_t>(HG) * pre_tail(b) + static_cast<int64_t>(hg) * nt;
                    unit_info[u].y = seg;
                    unit_info[u].z = static_cast<int>(t0 / kChunkStages);
                    unit_info[u].w = static_cast<int>(nt / kChunkStages);
                }
            } else {
                slot_of_piece = static_cast<int>(dyn_base + (seg - C) + u);
            }
            if (new_k && st == n - 1) flags |= kFlagAppend;  // position ctx - 1 is in this stage
            meta = min(kStageTokens, ctx - pos0) | flags | in_blk << 16;
            if constexpr (C8) {  // this stage's (block, head) scales, 0 for a block that will be skipped
                float *dst = bscl + (buf * 32 + lane) * 2 * HPC;
                const bool ok_id = id >= 0 && id < num_blocks;
                const int64_t base = (static_cast<int64_t>(id) * HG + hg) * HPC;
#pragma unroll
                for (int e = 0; e < HPC; ++e) {
                    dst[e] = ok_id ? __ldg(k_scale + base + e) : 0.f;
                    dst[HPC + e] = ok_id ? __ldg(v_scale + base + e) : 0.f;
                }
            }
        };
        // batch bookkeeping (warp-uniform)
        int64_t c_sb = 0, c_se = 0, c_lo = 0, c_hi = 0;
        int c_seg = -1;
        int cb = 0, chg = 0, cmeta = 0, cid = -1, cslot = 0;  // this lane's stage of the current batch
        int64_t static_next = s0;                   // next static stage not yet batched
        // the next batch: static stages first, then chunks of the dynamic region
        // (a ticket from the counter)
        auto next_batch = [&](int64_t &sb, int64_t &se, int64_t &lo, int64_t &hi, int &seg) -> bool {
            if (static_next < s1) {
                sb = static_next;
                se = min(static_next + 32, s1);
                lo = s0;
                hi = s1;
                seg = c;
                static_next = se;
                return true;
            }
            uint32_t k = 0;
            if (lane == 0) k = atomicAdd(chunk_ctr, 1u);
            k = __shfl_sync(0xffffffffu, k, 0);
            if (k >= K) return false;
            sb = static_cast<int64_t>(k) * kChunkStages;  // in the dynamic region
            se = sb + kChunkStages;
            lo = sb;
            hi = se;
            seg = C + static_cast<int>(k);
            return true;
        };
        int64_t n_sb = 0, n_se = 0, n_lo = 0, n_hi = 0;
        int n_seg = 0;
        bool have = next_batch(c_sb, c_se, c_lo, c_hi, c_seg);
        if (have) describe(c_sb, c_se, c_lo, c_hi, c_seg, cb, chg, cmeta, cid, cslot, cbuf);
        g_b = -1;  // the guess covers the first batch only
        bool aborted = false;
        int64_t issued = 0;
        while (have && !aborted) {
            // A static batch is described while the one before it is issued, as
            // soon as that one's first STAGES stages are out (the most that can be
            // in flight before the producer waits for a free slot), so its
            // block-id loads stay in flight meanwhile and the launch's first bulk
            // copies do not wait for them.  A dynamic chunk is claimed only when
            // kGrabAhead stages of the current batch remain, so that chunks go to
            // the CTAs that actually run out of work.
            int nb = 0, nhg = 0, nmeta = 0, nid = -1, nslot = 0;
            bool have_next = false, decided = false;
            const int cnt = static_cast<int>(c_se - c_sb);
            const int ahead_at = static_next < s1 ? min(cnt - 1, STAGES) : cnt - kGrabAhead;
            for (int j = 0; j < cnt; ++j) {
                if (!decided && j >= ahead_at) {
                    have_next = next_batch(n_sb, n_se, n_lo, n_hi, n_seg);
                    if (have_next) describe(n_sb, n_se, n_lo, n_hi, n_seg, nb, nhg, nmeta, nid, nslot, cbuf ^ 1);
                    decided = true;
                }
                const int b = __shfl_sync(0xffffffffu, cb, j), hg = __shfl_sync(0xffffffffu, chg, j);
                int meta = __shfl_sync(0xffffffffu, cmeta, j);
                int id = __shfl_sync(0xffffffffu, cid, j);
                const int pslot = __shfl_sync(0xffffffffu, cslot, j);
                // Early copies: the next one is this stage's (same block, row and
                // head group, no append) or its slot is skipped.
                while (issued < n_early) {
                    const int e = static_cast<int>(issued);
                    const int eid = __shfl_sync(0xffffffffu, e_id, e), ehg = __shfl_sync(0xffffffffu, e_hg, e);
                    const int erow = __shfl_sync(0xffffffffu, e_row, e);
                    if (eid == id && ehg == hg && erow == (meta >> 16) && !(meta & kFlagAppend)) break;
                    if (lane == 0) {
                        info[e] = make_int4(-2, 0, 0, 0);
                        mbar_arrive(bar0 + 8 * e);
                    }
                    issued = e + 1;
                }
                const int64_t i = issued;
                const bool early = i < n_early;  // this stage's bulk copy is in flight already
                const int slot = static_cast<int>(i % STAGES);
                const uint32_t full = bar0 + 8 * slot, empty = bar0 + 8 * (STAGES + slot);
                if ((meta & kFlagAppend) && id >= 0 && id < num_blocks) {
                    // Append: the step's new K/V rows of these HPC heads go to the
                    // cache row of position ctx - 1 before the bulk copy reads it
                    // back (the generic-proxy stores are ordered before the
                    // async-proxy load by fence.proxy.async).  Lane l moves dims
                    // 4l .. 4l + 3 of every head (8 bytes of the 16-bit row).
                    const int64_t row = static_cast<int64_t>(id) * bs + (meta >> 16) + ((meta & 0xff) - 1);
                    const int64_t src = (static_cast<int64_t>(b) * HG + hg) * HPC * kFastHeadDim;
                    const int64_t dst = (row * HG + hg) * HPC * kFastHeadDim;  // elements (16-bit) or codes
                    const int2 *sk = reinterpret_cast<const int2 *>(new_k + src);
                    const int2 *sv = reinterpret_cast<const int2 *>(new_v + src);
                    int2 tk[HPC], tv[HPC];  // HPC heads x 256 bytes = HPC x 32 lanes x 8 bytes
#pragma unroll
                    for (int e = 0; e < HPC; ++e) {
                        tk[e] = __ldg(sk + e * 32 + lane);
                        tv[e] = __ldg(sv + e * 32 + lane);
                    }
                    if constexpr (C8) {
                        // 8-bit cache: each head's four values become four codes
                        // under that head's existing (block, head) scale, loaded
                        // with this stage's description (the store kernels'
                        // encoding: x / s in binary32, round to nearest even).
                        __syncwarp();  // the describing lane wrote the scales
                        const float *sc = bscl + (cbuf * 32 + j) * 2 * HPC;  // [K: HPC][V: HPC]
                        uint8_t *dk = reinterpret_cast<uint8_t *>(k_cache_w) + dst;
                        uint8_t *dv = reinterpret_cast<uint8_t *>(v_cache_w) + dst;
#pragma unroll
                        for (int e = 0; e < HPC; ++e) {
                            const T *xk = reinterpret_cast<const T *>(&tk[e]);
                            const T *xv = reinterpret_cast<const T *>(&tv[e]);
                            const float s_k = sc[e], s_v = sc[HPC + e];
                            constexpr bool I8 = FMT == kCodeInt8;
                            const uint32_t ck = q8_encode2<I8>(to_f32(xk[0]), to_f32(xk[1]), s_k) |
                                                q8_encode2<I8>(to_f32(xk[2]), to_f32(xk[3]), s_k) << 16;
                            const uint32_t cv = q8_encode2<I8>(to_f32(xv[0]), to_f32(xv[1]), s_v) |
                                                q8_encode2<I8>(to_f32(xv[2]), to_f32(xv[3]), s_v) << 16;
                            *reinterpret_cast<uint32_t *>(dk + e * kFastHeadDim + 4 * lane) = ck;
                            *reinterpret_cast<uint32_t *>(dv + e * kFastHeadDim + 4 * lane) = cv;
                        }
                    } else {
                        int2 *dk = reinterpret_cast<int2 *>(k_cache_w + dst);
                        int2 *dv = reinterpret_cast<int2 *>(v_cache_w + dst);
#pragma unroll
                        for (int e = 0; e < HPC; ++e) {
                            dk[e * 32 + lane] = tk[e];
                            dv[e * 32 + lane] = tv[e];
                        }
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                }
                int ok = 1;
                if (lane == 0 && i >= STAGES) ok = mbar_wait(empty, ((i / STAGES) - 1) & 1, deadline) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    aborted = true;
                    break;
                }
                if (lane == 0) {
                    if (id < 0 || id >= num_blocks) {  // skip the block: its rows count as masked
                        id = -1;
                        bad = true;
                        meta &= ~0xff;
                    }
                    info[slot] = make_int4(b, hg, meta & 0xffff, pslot);
                    if constexpr (C8) {
                        const float *srcs = bscl + (cbuf * 32 + j) * 2 * HPC;
#pragma unroll
                        for (int e = 0; e < 2 * HPC; ++e) scl[slot * 2 * HPC + e] = srcs[e];
                    }
                    if (early) {
                        mbar_arrive(full);  // its bytes were expected when the copy left
                    } else if (id >= 0) {
                        const int slot_row = id * bs + (meta >> 16);
                        const uint32_t dst = tiles + slot * L::kStageBytes;
                        const int z = C8 ? hg * HPC : 2 * hg * HPC;  // first head (C8) or half-row of the box
                        mbar_arrive_expect_tx(full, L::kStageBytes);
                        if (kKvEvictFirst) {
                            tma_load_3d_hint(dst, &tm_k, 0, slot_row, z, full, kv_policy);
                            tma_load_3d_hint(dst + L::kTileBytes, &tm_v, 0, slot_row, z, full, kv_policy);
                        } else {
                            tma_load_3d(dst, &tm_k, 0, slot_row, z, full);
                            tma_load_3d(dst + L::kTileBytes, &tm_v, 0, slot_row, z, full);
                        }
                    } else {
                        mbar_arrive(full);  // nothing to load: the consumers mask the whole stage
                    }
                }
                issued = i + 1;
                __syncwarp();
            }
            have = have_next;
            c_sb = n_sb; c_se = n_se; c_lo = n_lo; c_hi = n_hi; c_seg = n_seg;
            cb = nb; chg = nhg; cmeta = nmeta; cid = nid; cslot = nslot;
            cbuf ^= 1;
        }
        while (!aborted && issued < n_early) {  // early copies no stage claimed (none, when the guess holds)
            if (lane == 0) {
                info[issued] = make_int4(-2, 0, 0, 0);
                mbar_arrive(bar0 + 8 * static_cast<int>(issued));
            }
            ++issued;
        }
        if (lane == 0) {
            if (!aborted) {
                // Tell the consumers there is no more work: a stage with b = -1.
                // They consume every real stage before it, so every bulk copy has
                // landed by the time they leave.
                const int64_t i = issued;
                const int slot = static_cast<int>(i % STAGES);
                if (i < STAGES || mbar_wait(bar0 + 8 * (STAGES + slot), ((i / STAGES) - 1) & 1, deadline)) {
                    info[slot] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(bar0 + 8 * slot);
                } else {
                    aborted = true;
                }
            }
            if (aborted) {
                *abort_flag = 1;
                if (err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
                // No bulk copy may still be writing shared memory when the CTA exits.
                for (int64_t i = issued - STAGES > 0 ? issued - STAGES : 0; i < issued; ++i)
                    if (!mbar_wait(bar0 + 8 * (i % STAGES), (i / STAGES) & 1, deadline) && err_flag)
                        atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
            }
        }
        if (bad && err_flag) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
        return;
    }

    // ---------------------------------------------------------------- consumer warp
    const int g = lane >> 2, t = lane & 3;
    const int mi = lane >> 3, r = lane & 7;
    // 16-bit caches: this head's rows of the stage tile; C8: the warp's own
    // widened tile (the same [2 halves][16 tokens][128 B] swizzled layout)
    const uint32_t head_off = C8 ? 0u : static_cast<uint32_t>(warp) * 2 * kStageTokens * 128;
    uint32_t k_off[8], v_off[8], v8_off[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // C8 V: lane l addresses row (l & 7) + 8((l >> 3) & 1), chunk 2j + (l >> 4)
        const int tok = r + 8 * (mi & 1);
        v8_off[j] = static_cast<uint32_t>(tok) * 128 + (((2 * j + (mi >> 1)) ^ (tok & 7)) << 4);
    }
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        {
            const int tok = r + 8 * (mi & 1);
            const int c16 = 2 * cc + (mi >> 1);
            k_off[cc] = head_off + ((c16 >> 3) * kStageTokens + tok) * 128 + (((c16 & 7) ^ r) << 4);
        }
        {
            const int tok = r + 8 * (mi >> 1);
            const int c16 = 2 * cc + (mi & 1);
            v_off[cc] = head_off + ((c16 >> 3) * kStageTokens + tok) * 128 + (((c16 & 7) ^ r) << 4);
        }
    }
    uint32_t qf[8][2];
    int q_b = -1, q_hg = -1;  // whose query heads qf holds
    auto load_q = [&](int b, int hg) {
        const int hk = hg * HPC + warp;
        const bool live = g < G;
        const uint32_t *q32 = reinterpret_cast<const uint32_t *>(
            q + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(hk) * G + (live ? g : 0)) * kFastHeadDim);
        if constexpr (C8) {
            // The 8-bit score MMAs take K fragments straight from the codes: in
            // MMA kc, lane t's k positions {2t, 2t+1, 2t+8, 2t+9} stand for dims
            // 32t + 4kc + {0, 1, 2, 3}, so q is read in that order (f16 MMAs).
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 v = live ? __ldg(reinterpret_cast<const uint4 *>(q32 + 16 * t) + j) : make_uint4(0, 0, 0, 0);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 2; ++e) {  // words 2e, 2e + 1 = dims 32t + 4(2j + e) + {0, 1}, {2, 3}
                    uint32_t lo = w[2 * e], hi = w[2 * e + 1];
                    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                        lo = bf16x2_to_f16x2(lo);
                        hi = bf16x2_to_f16x2(hi);
                    }
                    qf[2 * j + e][0] = lo;
                    qf[2 * j + e][1] = hi;
                }
            }
        } else {
#pragma unroll
            for (int kc = 0; kc < 8; ++kc) {
                qf[kc][0] = live ? __ldg(q32 + kc * 8 + t) : 0u;
                qf[kc][1] = live ? __ldg(q32 + kc * 8 + 4 + t) : 0u;
            }
        }
        q_b = b;
        q_hg = hg;
    };
    if (s0 < s1) {  // the first stage of the static slice is known now: fetch its queries early
        int b, hg, st;
        locate_stage(pre_static, B, HG, s0, b, hg, st);
        load_q(b, hg);
    }
    float o[8][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    for (int64_t i = 0;; ++i) {
        const int slot = static_cast<int>(i % STAGES);
        if (!mbar_wait(bar0 + 8 * slot, (i / STAGES) & 1, deadline) || *abort_flag) {
            if (lane == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
            return;
        }
        const int4 inf = info[slot];
        const int b = inf.x, hg = inf.y, meta = inf.z, pslot = inf.w;
        if (b == -1) break;  // no more work
        if (b < 0) {         // an early copy no stage claimed: release the slot
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + 8 * (STAGES + slot));
            continue;
        }
        const int nvalid = meta & 0xff;
        const int hk = hg * HPC + warp;
        if (meta & kFlagFirst) {
            if (b != q_b || hg != q_hg) load_q(b, hg);
#pragma unroll
            for (int dc = 0; dc < 8; ++dc)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[dc][e] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }
        uint32_t kt, vt;  // K / V tiles the ldmatrix offsets apply to
        float sl = scale_log2, sv = 1.f;
        if constexpr (C8) {
            // this head's 8-bit rows [16 tokens][128 B] of K and of V, and their scales
            kt = tiles + slot * L::kStageBytes + static_cast<uint32_t>(warp) * kStageTokens * 128;
            vt = kt + L::kTileBytes;
            sl = scale_log2 * scl[slot * 2 * HPC + warp];
            sv = scl[slot * 2 * HPC + HPC + warp];
            if (nvalid < kStageTokens) {  // V rows past the valid ones: zeros (their codes may be NaN)
                const int nbad = kStageTokens - nvalid;
                for (int idx = lane; idx < nbad * 8; idx += 32) {
                    const uint32_t addr = vt + (nvalid + (idx >> 3)) * 128 + (idx & 7) * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
                }
                __syncwarp();
            }
        } else {
            kt = tiles + slot * L::kStageBytes;
            vt = kt + L::kTileBytes;
            if (nvalid < kStageTokens) {
                // Rows past the context (or of a skipped block) may hold anything,
                // NaN included: zero this head's V rows so that 0 * row stays 0.
                const int nbad = kStageTokens - nvalid;
                for (int idx = lane; idx < nbad * 16; idx += 32) {
                    const int tok = nvalid + (idx >> 4);
                    const int half = (idx >> 3) & 1;
                    const int chunk = idx & 7;
                    const uint32_t addr = vt + head_off + (half * kStageTokens + tok) * 128 + chunk * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
                }
                __syncwarp();
            }
        }
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (C8) {
            // Rows g and g + 8 of this head's codes, bytes 32t .. 32t + 31 (chunks
            // 2t, 2t + 1 at their swizzled places): word kc of a row gives MMA
            // kc's k positions (2t, 2t+1) and (2t+8, 2t+9).
            const uint32_t k8 = kt;
            uint32_t wr[2][8];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = g + 8 * rr;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(wr[rr][4 * h2]), "=r"(wr[rr][4 * h2 + 1]), "=r"(wr[rr][4 * h2 + 2]),
                                   "=r"(wr[rr][4 * h2 + 3])
                                 : "r"(k8 + static_cast<uint32_t>(row) * 128 + (((2 * t + h2) ^ (row & 7)) << 4)));
            }
#pragma unroll
            for (int kc = 0; kc < 8; ++kc) {
                uint32_t a[4];
                codes4_to_f16x4<FMT, false>(wr[0][kc], a[0], a[2]);
                codes4_to_f16x4<FMT, false>(wr[1][kc], a[1], a[3]);
                H::mma(sc, a, qf[kc][0], qf[kc][1]);
            }
        } else {
#pragma unroll
            for (int kc = 0; kc < 8; ++kc) {
                uint32_t a[4];
                ldsm_x4(kt + k_off[kc], a);
                H::mma(sc, a, qf[kc][0], qf[kc][1]);
            }
        }
        const bool vg = g < nvalid, vg8 = g + 8 < nvalid;
        const float x0 = vg ? sc[0] * sl : -INFINITY;
        const float x1 = vg ? sc[1] * sl : -INFINITY;
        const float x2 = vg8 ? sc[2] * sl : -INFINITY;
        const float x3 = vg8 ? sc[3] * sl : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float p0 = fast_exp2(x0 - base0), p1 = fast_exp2(x1 - base1);
        const float p2 = fast_exp2(x2 - base0), p3 = fast_exp2(x3 - base1);
        const float a0 = fast_exp2(m0 - base0), a1 = fast_exp2(m1 - base1);
        m0 = mn0;
        m1 = mn1;
        l0 = l0 * a0 + (p0 + p2);
        l1 = l1 * a1 + (p1 + p3);
#pragma unroll
        for (int dc = 0; dc < 8; ++dc) {
            o[dc][0] *= a0;
            o[dc][1] *= a1;
            o[dc][2] *= a0;
            o[dc][3] *= a1;
        }
        // C8: the V scale rides on P (sv = 1 for 16-bit caches); the sums l use P itself
        const uint32_t pb0 = movmatrix_trans(H::pack(p0 * sv, p1 * sv));
        const uint32_t pb1 = movmatrix_trans(H::pack(p2 * sv, p3 * sv));
        if constexpr (C8) {
            // V^T fragments straight from the codes: ldmatrix.trans of the tile
            // read as b16 gives lane (g, t) the bytes (V[2t][2g], V[2t][2g+1],
            // V[2t+1][2g], V[2t+1][2g+1]) of a 16-dim chunk; a byte permute
            // pairs them per dim, so MMA dc's row g is dim 16dc + 2g and row
            // g + 8 is dim 16dc + 2g + 1 (the output mapping below follows).
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // chunks 2j and 2j + 1: MMAs 2j, 2j + 1
                uint32_t w[4];
                ldsm_x4_trans(vt + v8_off[j], w);  // (tokens 0-7 | 8-15) x (chunk 2j | 2j + 1)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint32_t a[4];
                    codes4_to_f16x4<FMT, true>(w[2 * e], a[0], a[1]);
                    codes4_to_f16x4<FMT, true>(w[2 * e + 1], a[2], a[3]);
                    H::mma(o[2 * j + e], a, pb0, pb1);
                }
            }
        } else {
#pragma unroll
            for (int dc = 0; dc < 8; ++dc) {
                uint32_t a[4];
                ldsm_x4_trans(vt + v_off[dc], a);
                H::mma(o[dc], a, pb0, pb1);
            }
        }
        if (nvalid < kStageTokens) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(bar0 + 8 * (STAGES + slot));

        if (meta & kFlagLast) {
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
                l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
            }
            const int hA = 2 * t, hB = 2 * t + 1;
            if (meta & kFlagWhole) {
                const int64_t qhead0 = static_cast<int64_t>(b) * Hq + static_cast<int64_t>(hk) * G;
                const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
                for (int dc = 0; dc < 8; ++dc) {
                    const int d0 = C8 ? dc * 16 + 2 * g : dc * 16 + g, d1 = C8 ? d0 + 1 : d0 + 8;
                    if (hA < G) {
                        T *dst = out + (qhead0 + hA) * kFastHeadDim;
                        dst[d0] = from_f32<T>(o[dc][0] * inv0);
                        dst[d1] = from_f32<T>(o[dc][2] * inv0);
                    }
                    if (hB < G) {
                        T *dst = out + (qhead0 + hB) * kFastHeadDim;
                        dst[d0] = from_f32<T>(o[dc][1] * inv1);
                        dst[d1] = from_f32<T>(o[dc][3] * inv1);
                    }
                }
            } else {
                const int64_t piece = static_cast<int64_t>(pslot) * HPC + warp;  // * G + head
#pragma unroll
                for (int dc = 0; dc < 8; ++dc) {
                    const int d0 = C8 ? dc * 16 + 2 * g : dc * 16 + g, d1 = C8 ? d0 + 1 : d0 + 8;
                    if (hA < G) {
                        float *dst = o_piece + (piece * G + hA) * kFastHeadDim;
                        dst[d0] = o[dc][0];
                        dst[d1] = o[dc][2];
                    }
                    if (hB < G) {
                        float *dst = o_piece + (piece * G + hB) * kFastHeadDim;
                        dst[d0] = o[dc][1];
                        dst[d1] = o[dc][3];
                    }
                }
                if (g == 0) {
                    if (hA < G) ml_piece[piece * G + hA] = make_float2(m0, l0);
                    if (hB < G) ml_piece[piece * G + hB] = make_float2(m1, l1);
                }
            }
        }
    }
}

// Merges the pieces of every split unit.  A row is one (unit, query head of
// the unit) pair; WPR warps of a CTA of 8 share a row, so a CTA covers 8 / WPR
// rows (the host picks WPR so that the grid stays near one wave: 8 warps per
// row for launches with few units and many pieces each, fewer when units are
// many).  unit_info[u] = (first static slice, last static slice, first chunk,
// chunk count) gives the unit's pieces: slot (c + u) for its static slices and
// (dyn_base + k + u) for its chunks.  The kernel makes two dependent rounds of
// loads: the unit's context length and unit_info, then every piece's (max,
// sum) pair and output row, kMergeInFlight per warp at once.  Each warp folds
// its pieces into a running (max, sum, row) (lanes over the 128 dims as
// float4); the row's warps meet in shared memory.  The CTA is small (4 KB of
// shared memory) so that it fits beside two main-pass CTAs on an SM and is
// already resident when the main pass ends.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeInFlight = 8;  // pieces per warp per round
constexpr int kMergeWaveCtas = 608;   // grid target: 4 merge CTAs per SM (beat 8 per SM on GB300)

template <typename T, int WPR>
__global__ void __launch_bounds__(kMergeThreads)
stream_combine_kernel(T *__restrict__ out, const float *__restrict__ o_piece, const float2 *__restrict__ ml_piece,
                      const int4 *__restrict__ unit_info, const int32_t *__restrict__ context_lens, int32_t Hq,
                      int32_t HG, int32_t HU, int32_t bs, int32_t max_blocks, int32_t max_ctx, int32_t num_ctas,
                      int64_t dyn_base, int64_t max_slots, int64_t rows) {
    constexpr int RPC = kMergeWarps / WPR;  // rows per CTA
    __shared__ float4 red[kMergeWarps][32];
    __shared__ float2 wml[kMergeWarps];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % WPR;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * RPC + warp / WPR;
    int u = 0, j = 0, b = 0, hg = 0, f = 0, np = 0, n_static = 0, k0 = 0;
    if (row < rows) {
        const int r = static_cast<int>(row);  // rows = units * HU stays far below 2^31
        u = r / HU;
        j = r - u * HU;
        b = u / HG;
        hg = u - b * HG;
        const int ctx = context_lens[b];
        const int4 ui = unit_info[u];
        const int l = ui.y, nk = ui.w;
        f = ui.x;
        k0 = ui.z;
        // nothing to do: an empty or invalid context (zero row written by the
        // main pass), one piece (the main pass wrote the output), or unit_info
        // left inconsistent by an aborted main pass (PKV_ERRBIT_TIMEOUT is set)
        const bool work = context_ok(ctx, max_ctx, bs, max_blocks) && ctx != 0 && !(f == l && nk == 0) &&
                          f >= 0 && l >= f && l < num_ctas && k0 >= 0 && nk >= 0 &&
                          dyn_base + k0 + nk + u <= max_slots;
        if (work) {
            n_static = l - f + 1;
            np = n_static + nk;
        }
    }
    auto row_of = [&](int k) -> int64_t {
        const int64_t slot = k < n_static ? static_cast<int64_t>(f + k) + u : dyn_base + k0 + (k - n_static) + u;
        return slot * HU + j;
    };
    float m_w = -INFINITY, l_w = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int kb = sub; kb < np; kb += WPR * kMergeInFlight) {
        float4 v[kMergeInFlight];
        float2 ml[kMergeInFlight];
#pragma unroll
        for (int uu = 0; uu < kMergeInFlight; ++uu) {
            const int k = kb + WPR * uu;
            if (k < np) {
                const int64_t r = row_of(k);
                v[uu] = __ldg(reinterpret_cast<const float4 *>(o_piece + r * kFastHeadDim) + lane);
                ml[uu] = __ldg(ml_piece + r);
            } else {
                v[uu] = make_float4(0.f, 0.f, 0.f, 0.f);
                ml[uu] = make_float2(-INFINITY, 0.f);
            }
        }
        float mn = m_w;
#pragma unroll
        for (int uu = 0; uu < kMergeInFlight; ++uu) mn = fmaxf(mn, ml[uu].x);
        if (mn == -INFINITY) continue;  // nothing but empty pieces so far
        const float sc = exp2f(m_w - mn);  // 0 while m_w is still -inf
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
        l_w *= sc;
#pragma unroll
        for (int uu = 0; uu < kMergeInFlight; ++uu) {
            const float w = exp2f(ml[uu].x - mn);  // 0 for an empty piece (max -inf)
            acc.x = fmaf(w, v[uu].x, acc.x);
            acc.y = fmaf(w, v[uu].y, acc.y);
            acc.z = fmaf(w, v[uu].z, acc.z);
            acc.w = fmaf(w, v[uu].w, acc.w);
            l_w = fmaf(w, ml[uu].y, l_w);
        }
        m_w = mn;
    }
    if constexpr (WPR > 1) {
        red[warp][lane] = acc;
        if (lane == 0) wml[warp] = make_float2(m_w, l_w);
        __syncthreads();
        if (sub != 0 || np == 0) return;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < WPR; ++ww) M = fmaxf(M, wml[warp + ww].x);
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        l_w = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int ww = 0; ww < WPR; ++ww) {
                const float w = exp2f(wml[warp + ww].x - M);
                const float4 x = red[warp + ww][lane];
                acc.x = fmaf(w, x.x, acc.x);
                acc.y = fmaf(w, x.y, acc.y);
                acc.z = fmaf(w, x.z, acc.z);
                acc.w = fmaf(w, x.w, acc.w);
                l_w = fmaf(w, wml[warp + ww].y, l_w);
            }
        }
    } else if (np == 0) {
        return;
    }
    const float inv = l_w > 0.f ? 1.f / l_w : 0.f;
    T *dst = out + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(hg) * HU + j) * kFastHeadDim + 4 * lane;
    dst[0] = from_f32<T>(acc.x * inv);
    dst[1] = from_f32<T>(acc.y * inv);
    dst[2] = from_f32<T>(acc.z * inv);
    dst[3] = from_f32<T>(acc.w * inv);
}

// ----------------------------------------------------------------------------- append (other paths)
// The step's new K/V rows for the paths that do not append inside the
// attention kernel: row ctx - 1 of every sequence with a valid, non-empty
// context receives key[b] / value[b] (the slot rule of "Step 1: slot_mapping
// and store_kvcache").  One warp per (sequence, segment of 32 x 4 vectors).
constexpr int kAppendThreads = 256;

template <typename V>
__global__ void __launch_bounds__(kAppendThreads)
append_kv_kernel(const char *__restrict__ key, const char *__restrict__ value, char *__restrict__ k_cache,
                 char *__restrict__ v_cache, const int32_t *__restrict__ block_tables, int32_t max_blocks,
                 const int32_t *__restrict__ context_lens, int32_t B, int32_t bs, int32_t num_blocks,
                 int32_t max_ctx, int64_t row_bytes, int32_t *__restrict__ err_flag) {
    pdl_wait();
    pdl_trigger();
    constexpr int64_t kSeg = 32 * 4 * static_cast<int64_t>(sizeof(V));
    const int lane = threadIdx.x & 31;
    const int64_t nseg = (row_bytes + kSeg - 1) / kSeg;
    const int64_t items = static_cast<int64_t>(B) * nseg;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kAppendThreads / 32);
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * (kAppendThreads / 32) + (threadIdx.x >> 5); it < items;
         it += warps) {
        const int b = static_cast<int>(it / nseg);
        const int64_t seg = it - static_cast<int64_t>(b) * nseg;
        const int ctx = context_lens[b];
        if (ctx <= 0 || !context_ok(ctx, max_ctx, bs, max_blocks)) continue;  // the attention flags it
        const int p = ctx - 1;
        const int32_t blk = block_tables[static_cast<int64_t>(b) * max_blocks + p / bs];
        if (blk < 0 || blk >= num_blocks) {
            if (lane == 0 && seg == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
            continue;
        }
        const int64_t src = static_cast<int64_t>(b) * row_bytes + seg * kSeg;
        const int64_t dst = (static_cast<int64_t>(blk) * bs + p % bs) * row_bytes + seg * kSeg;
        V kv[4], vv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t off = (static_cast<int64_t>(u) * 32 + lane) * static_cast<int64_t>(sizeof(V));
            if (seg * kSeg + off < row_bytes) {
                kv[u] = *reinterpret_cast<const V *>(key + src + off);
                vv[u] = *reinterpret_cast<const V *>(value + src + off);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t off = (static_cast<int64_t>(u) * 32 + lane) * static_cast<int64_t>(sizeof(V));
            if (seg * kSeg + off < row_bytes) {
                *reinterpret_cast<V *>(k_cache + dst + off) = kv[u];
                *reinterpret_cast<V *>(v_cache + dst + off) = vv[u];
            }
        }
    }
}

// ----------------------------------------------------------------------------- host side
// 8-bit code pool [num_slots, Hkv, 128] of bytes viewed as (128 codes,
// num_slots, Hkv heads): one 128-byte row per (token, head), HPC heads per box.
pkv_status make_kv_map_8bit(CUtensorMap *map, const void *pool, int64_t num_slots, int Hkv, int hpc) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(PKV_ERR_CUDA, "decode: cuTensorMapEncodeTiled entry point unavailable");
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kFastHeadDim), static_cast<cuuint64_t>(num_slots),
                                static_cast<cuuint64_t>(Hkv)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Hkv) * kFastHeadDim, kFastHeadDim};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kFastHeadDim), kStageTokens, static_cast<cuuint32_t>(hpc)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(PKV_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

// cudaFuncSetAttribute once per (kernel, device); `done` is the caller's
// per-kernel bitmask of devices already configured.
template <typename K>
cudaError_t ensure_smem(K kernel, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

struct DecodeArgs {
    void *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables;
    int32_t max_blocks;
    const int32_t *context_lens;
    int32_t B, Hq, Hkv, d, bs, num_blocks, max_ctx;
    float scale;
    float *o_part;
    float2 *ml_part;
    int4 *unit_info;  // work-balanced schedule only
    int32_t *ws_meta;
    uint32_t *chunk_ctr;
    const void *new_k, *new_v;  // the step's new K/V rows [B, Hkv, d] to append first, or null
    const float *k_scale, *v_scale;  // 8-bit caches: scales [num_blocks, Hkv]; null for 16-bit caches
    int32_t *err;
    cudaStream_t stream;
    int32_t codes = kCode16;  // the cache's code format (CacheCode)
};

pkv_status launch_append(const DecodeArgs &a, int64_t es) {
    const int64_t row_bytes = static_cast<int64_t>(a.Hkv) * a.d * es;
    auto kc = static_cast<char *>(const_cast<void *>(a.k_cache));
    auto vc = static_cast<char *>(const_cast<void *>(a.v_cache));
    auto kk = static_cast<const char *>(a.new_k);
    auto vv = static_cast<const char *>(a.new_v);
    const bool v16 = row_bytes % 16 == 0 && aligned(kc, 16) && aligned(vc, 16) && aligned(kk, 16) && aligned(vv, 16);
    const bool v8 = row_bytes % 8 == 0 && aligned(kc, 8) && aligned(vc, 8) && aligned(kk, 8) && aligned(vv, 8);
    const int64_t vec = v16 ? 16 : v8 ? 8 : es;
    const int64_t items = static_cast<int64_t>(a.B) * ((row_bytes + 128 * vec - 1) / (128 * vec));
    int64_t grid = (items + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
    if (grid > 1024) grid = 1024;
    if (grid < 1) grid = 1;
    cudaError_t e;
#define PKV_APPEND(V) \
    launch_pdl(kPdlStore, append_kv_kernel<V>, dim3(static_cast<unsigned>(grid)), dim3(kAppendThreads), 0, a.stream, kk, \
               vv, kc, vc, a.block_tables, a.max_blocks, a.context_lens, a.B, a.bs, a.num_blocks, a.max_ctx, row_bytes, a.err)
    switch (vec) {
    case 16: e = PKV_APPEND(int4); break;
    case 8: e = PKV_APPEND(int2); break;
    case 4: e = PKV_APPEND(int); break;
    default: e = PKV_APPEND(short); break;
    }
#undef PKV_APPEND
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

// CTAs of the one-wave work-balanced grid on the current device:
// (resident CTAs per SM) x (SMs), capped by the workspace bound.
template <typename K>
int stream_ctas(K kernel, int threads, int smem, std::atomic<int> *per_device) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = per_device[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    c = per_sm * sms;
    if (c > kMaxStreamCtas) c = kMaxStreamCtas;
    if (c > 0) per_device[dev].store(c, std::memory_order_release);
    return c;
}

template <typename T, int HPC, int STAGES, int FMT>
struct StreamLaunch {
    static std::atomic<int> ctas[64];
    static std::atomic<uint64_t> configured;
    static int grid() {
        using L = StreamSmem<HPC, STAGES, FMT != kCode16>;
        if (ensure_smem(decode_stream_kernel<T, HPC, STAGES, FMT>, L::kAlloc, configured) != cudaSuccess) return 0;
        return stream_ctas(decode_stream_kernel<T, HPC, STAGES, FMT>, (HPC + 1) * 32, L::kAlloc, ctas);
    }
};
template <typename T, int HPC, int STAGES, int FMT> std::atomic<int> StreamLaunch<T, HPC, STAGES, FMT>::ctas[64];
template <typename T, int HPC, int STAGES, int FMT>
std::atomic<uint64_t> StreamLaunch<T, HPC, STAGES, FMT>::configured{0};

// Warps per merge row: as many as keep the merge grid within about one wave.
inline int merge_warps_per_row(int64_t rows) {
    int wpr = kMergeWarps;
    while (wpr > 1 && rows * wpr > static_cast<int64_t>(kMergeWaveCtas) * kMergeWarps) wpr >>= 1;
    return wpr;
}

template <typename T>
cudaError_t launch_stream_combine(const DecodeArgs &a, const Plan &p, int C, int HG, int HU) {
    const int64_t units = static_cast<int64_t>(a.B) * HG;  // this launch's group (<= p.units)
    const int64_t rows = units * HU;
    const int wpr = merge_warps_per_row(rows);
    const int64_t rpc = kMergeWarps / wpr;
    const dim3 grid(static_cast<unsigned>((rows + rpc - 1) / rpc));
    auto kern = wpr == 8 ? stream_combine_kernel<T, 8>
              : wpr == 4 ? stream_combine_kernel<T, 4>
              : wpr == 2 ? stream_combine_kernel<T, 2>
                         : stream_combine_kernel<T, 1>;
    return launch_pdl(kPdlCombine, kern, grid, dim3(kMergeThreads), 0, a.stream, static_cast<T *>(a.out),
                      static_cast<const float *>(a.o_part), static_cast<const float2 *>(a.ml_part),
                      static_cast<const int4 *>(a.unit_info), a.context_lens, a.Hq, HG, HU, a.bs, a.max_blocks,
                      a.max_ctx, C, static_cast<int64_t>(kMaxStreamCtas + units),
                      static_cast<int64_t>(p.max_segments), rows);
}

template <typename T, int HPC, int STAGES, int FMT>
pkv_status launch_stream(const DecodeArgs &a, const Plan &p) {
    using L = StreamSmem<HPC, STAGES, FMT != kCode16>;
    CUtensorMap mk, mv;
    const int64_t slots = static_cast<int64_t>(a.num_blocks) * a.bs;
    pkv_status st = FMT != kCode16 ? make_kv_map_8bit(&mk, a.k_cache, slots, a.Hkv, HPC)
                        : make_kv_map(&mk, a.k_cache, Half16<T>::kTmaType, slots, a.Hkv, HPC);
    if (st != PKV_OK) return st;
    st = FMT != kCode16 ? make_kv_map_8bit(&mv, a.v_cache, slots, a.Hkv, HPC)
             : make_kv_map(&mv, a.v_cache, Half16<T>::kTmaType, slots, a.Hkv, HPC);
    if (st != PKV_OK) return st;
    const int C = StreamLaunch<T, HPC, STAGES, FMT>::grid();
    if (C <= 0) return set_error(PKV_ERR_CUDA, "decode: no resident CTA fits the work-balanced kernel");
    const int HG = a.Hkv / HPC, G = a.Hq / a.Hkv;
    cudaError_t e = launch_pdl(kPdlDecode, decode_stream_kernel<T, HPC, STAGES, FMT>, dim3(C), dim3((HPC + 1) * 32),
                               L::kAlloc, a.stream, mk, mv, static_cast<T *>(a.out), static_cast<const T *>(a.q),
                               a.block_tables, a.max_blocks, a.context_lens, a.B, a.Hq, G, HG, a.bs, a.num_blocks,
                               a.max_ctx, a.scale * kLog2e, a.o_part, a.ml_part, a.unit_info, a.ws_meta,
                               a.chunk_ctr, static_cast<const T *>(a.new_k), static_cast<const T *>(a.new_v),
                               static_cast<T *>(const_cast<void *>(a.k_cache)),
                               static_cast<T *>(const_cast<void *>(a.v_cache)), a.k_scale, a.v_scale, a.err);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    e = launch_stream_combine<T>(a, p, C, HG, HPC * G);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

// Pipeline depth per (heads per CTA, cache format): about 96 KB of stages and
// two CTAs per SM for 16-bit caches; 48 KB (32 KB for one head) and three
// CTAs per SM for 8-bit caches, whose consumers do more work per byte and need
// the extra warps to hide latency (measured: 181 vs 199 us on the LLaMA layer).
template <typename T>
pkv_status launch_stream_any(const DecodeArgs &a, const Plan &p) {
    if (a.codes == kCodeE4M3) {
        switch (p.hpc) {
        case 4: return launch_stream<T, 4, 3, kCodeE4M3>(a, p);
        case 2: return launch_stream<T, 2, 6, kCodeE4M3>(a, p);
        default: return launch_stream<T, 1, 8, kCodeE4M3>(a, p);
        }
    }
    if (a.codes == kCodeInt8) {
        switch (p.hpc) {
        case 4: return launch_stream<T, 4, 3, kCodeInt8>(a, p);
        case 2: return launch_stream<T, 2, 6, kCodeInt8>(a, p);
        default: return launch_stream<T, 1, 8, kCodeInt8>(a, p);
        }
    }
    switch (p.hpc) {
    case 4: return launch_stream<T, 4, 3, kCode16>(a, p);
    case 2: return launch_stream<T, 2, 6, kCode16>(a, p);
    default: return launch_stream<T, 1, 8, kCode16>(a, p);
    }
}

int stream_grid_for(pkv_dtype dt, int hpc) {
    if (dt == PKV_BF16) {
        switch (hpc) {
        case 4: return StreamLaunch<__nv_bfloat16, 4, 3, kCode16>::grid();
        case 2: return StreamLaunch<__nv_bfloat16, 2, 6, kCode16>::grid();
        default: return StreamLaunch<__nv_bfloat16, 1, 8, kCode16>::grid();
        }
    }
    switch (hpc) {
    case 4: return StreamLaunch<__half, 4, 3, kCode16>::grid();
    case 2: return StreamLaunch<__half, 2, 6, kCode16>::grid();
    default: return StreamLaunch<__half, 1, 8, kCode16>::grid();
    }
}

template <typename T, int HPC, int STAGES>
pkv_status launch_fast(const DecodeArgs &a, const Plan &p) {
    using L = FastSmem<HPC, STAGES>;
    CUtensorMap mk, mv;
    pkv_status st = make_kv_map(&mk, a.k_cache, Half16<T>::kTmaType, static_cast<int64_t>(a.num_blocks) * a.bs, a.Hkv, HPC);
    if (st != PKV_OK) return st;
    st = make_kv_map(&mv, a.v_cache, Half16<T>::kTmaType, static_cast<int64_t>(a.num_blocks) * a.bs, a.Hkv, HPC);
    if (st != PKV_OK) return st;
    auto kern = decode_fast_kernel<T, HPC, STAGES>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = ensure_smem(kern, L::kAlloc, configured);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "decode: smem attribute: %s", cudaGetErrorString(e));
    // At least one partition, so that zero-length contexts still get their zero rows.
    dim3 grid(p.nparts > 0 ? p.nparts : 1, a.Hkv / HPC, a.B);
    e = launch_pdl(kPdlDecode, kern, grid, dim3((HPC + 1) * 32), L::kAlloc, a.stream, mk, mv, static_cast<T *>(a.out),
                   static_cast<const T *>(a.q), a.block_tables, a.max_blocks, a.context_lens, a.Hq, a.Hq / a.Hkv,
                   a.bs, a.num_blocks, a.max_ctx, p.partition, p.nparts, a.scale * kLog2e, a.o_part, a.ml_part,
                   a.err);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

template <typename T>
pkv_status launch_fast_any(const DecodeArgs &a, const Plan &p) {
    switch (p.hpc) {
    case 4: return launch_fast<T, 4, 3>(a, p);
    case 2: return launch_fast<T, 2, 6>(a, p);
    default: return launch_fast<T, 1, 8>(a, p);
    }
}

template <typename T>
pkv_status launch_generic_and_combine(const DecodeArgs &a, const Plan &p, bool run_main) {
    if (run_main) {
        const size_t smem = (static_cast<size_t>(a.d) + p.partition + 32) * sizeof(float);
        auto kern = decode_generic_kernel<T>;
        static std::atomic<uint64_t> configured{0};
        cudaError_t e = ensure_smem(kern, static_cast<int>(48 * 1024), configured);
        if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "decode: smem attribute: %s", cudaGetErrorString(e));
        dim3 grid(p.nparts > 0 ? p.nparts : 1, a.Hq, a.B);
        e = launch_pdl(kPdlDecode, kern, grid, dim3(kGenThreads), smem, a.stream, static_cast<T *>(a.out),
                       static_cast<const T *>(a.q), static_cast<const T *>(a.k_cache),
                       static_cast<const T *>(a.v_cache), a.block_tables, a.max_blocks, a.context_lens, a.Hq, a.Hkv,
                       a.d, a.bs, a.num_blocks, a.max_ctx, p.partition, p.nparts, a.scale * kLog2e, a.o_part,
                       a.ml_part, a.err);
        if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    }
    if (p.nparts > 1) {
        cudaError_t e = launch_combine<T>(static_cast<T *>(a.out), a.o_part, a.ml_part, a.context_lens, a.Hq, a.B,
                                          a.d, a.bs, a.max_blocks, a.max_ctx, p.partition, p.nparts, a.stream);
        if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    }
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_paged_attention_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                            int32_t num_kv_heads, int32_t head_dim,
                                                            int32_t block_size, int32_t max_context_len,
                                                            pkv_dtype dtype) {
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        head_dim <= 0 || block_size <= 0 || max_context_len < 0 || dtype_bytes(dtype) == 0)
        return 0;
    // one size for 16-bit and 8-bit caches (their plans differ past 512 sequences)
    const size_t a = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, dtype).ws_bytes;
    const size_t b = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, dtype,
                               false, 0, true).ws_bytes;
    return a > b ? a : b;
}

extern "C" pkv_status pkv_paged_attention_decode_plan(int32_t num_seqs, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t head_dim,
                                                      int32_t block_size, int32_t max_context_len,
                                                      pkv_dtype dtype, int32_t *partition_tokens,
                                                      int32_t *num_partitions, int32_t *fast_path) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        head_dim <= 0 || block_size <= 0 || max_context_len < 0 || dtype_bytes(dtype) == 0)
        return set_error(PKV_ERR_INVALID_ARG, "decode plan: bad sizes");
    Plan p = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, dtype);
    if (partition_tokens) *partition_tokens = p.partition;
    if (num_partitions) *num_partitions = p.stream ? stream_grid_for(dtype, p.hpc) : p.nparts;
    if (fast_path) *fast_path = p.fast ? 1 : 0;
    return ok();
}

namespace pkv {
namespace {

// Sizes, dtype and pointers of a decode call, checked before anything else
// (the workspace is checked later, against the plan these sizes give).
pkv_status check_decode_args(const void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, int32_t max_context_len, pkv_dtype dtype) {
    if (dtype_bytes(dtype) == 0) return set_error(PKV_ERR_INVALID_ARG, "decode: unknown dtype %d", (int)dtype);
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || max_context_len < 0 || max_blocks_per_seq < 0)
        return set_error(PKV_ERR_INVALID_ARG, "decode: bad sizes");
    if (num_q_heads % num_kv_heads)
        return set_error(PKV_ERR_INVALID_ARG, "decode: num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                         num_q_heads, num_kv_heads);
    if (head_dim > 1024) return set_error(PKV_ERR_UNSUPPORTED, "decode: head_dim > 1024");
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return set_error(PKV_ERR_INVALID_ARG, "decode: num_blocks * block_size >= 2^31");
    if (num_seqs > 65535) return set_error(PKV_ERR_UNSUPPORTED, "decode: more than 65535 sequences in one call");
    if (num_seqs > 0 && (!out || !q || !context_lens || (max_blocks_per_seq > 0 && !block_tables) ||
                         (num_blocks > 0 && (!k_cache || !v_cache))))
        return set_error(PKV_ERR_INVALID_ARG, "decode: NULL pointer");
    return PKV_OK;
}

// Decode attention, with the step's new K/V rows appended first when new_k is
// not null (the fused decode step).
pkv_status decode_entry(void *out, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                        pkv_dtype dtype, void *workspace, size_t workspace_bytes, int32_t *err_flag, void *stream,
                        const void *new_k, const void *new_v, const float *k_scale = nullptr,
                        const float *v_scale = nullptr, int32_t codes = kCode16) {
    const int64_t es = dtype_bytes(dtype);
    const bool c8 = codes != kCode16;  // 8-bit caches with per-(block, head) scales
    const char *fmt = codes == kCodeInt8 ? "int8" : "fp8";
    pkv_status chk = check_decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                       max_context_len, dtype);
    if (chk != PKV_OK) return chk;
    if (num_seqs == 0) return ok();
    const bool append = new_k != nullptr || new_v != nullptr;
    if (append && (!new_k || !new_v || !aligned(new_k, es) || !aligned(new_v, es)))
        return set_error(PKV_ERR_INVALID_ARG, "decode append: key/value NULL or not aligned to the element size");
    Plan p = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, dtype, false, 0, c8);
    if (p.ws_bytes > 0 && (!workspace || workspace_bytes < p.ws_bytes || !aligned(workspace, 256)))
        return set_error(PKV_ERR_WORKSPACE, "decode: workspace needs %zu bytes (256-byte aligned), got %zu",
                         p.ws_bytes, workspace_bytes);
    if (!aligned(out, es) || !aligned(q, es) || (k_cache && !aligned(k_cache, es)) || (v_cache && !aligned(v_cache, es)))
        return set_error(PKV_ERR_INVALID_ARG, "decode: buffers not aligned to the element size");
    // The fast path additionally wants 16-byte aligned pools (TMA) and 4-byte aligned q.
    const bool fast = p.fast && num_blocks > 0 && aligned(k_cache, 16) && aligned(v_cache, 16) && aligned(q, 4);
    if (c8) {
        if (!fast || !p.stream || !aligned(q, 16) || (append && (!aligned(new_k, 8) || !aligned(new_v, 8))))
            return set_error(PKV_ERR_UNSUPPORTED,
                             "decode %s: needs fp16/bf16 q, head_dim 128, Hq/Hkv <= 8, block_size a multiple of "
                             "16, 16-byte aligned q and code pools (and 8-byte aligned key/value to append)",
                             fmt);
        if (!k_scale || !v_scale || !aligned(k_scale, 4) || !aligned(v_scale, 4))
            return set_error(PKV_ERR_INVALID_ARG, "decode %s: scales NULL or not 4-byte aligned", fmt);
    }
    if (p.fast && !fast) {
        // CUDA-core fallback with partitions that fit the workspace sized for the fast plan.
        const int64_t per_part = static_cast<int64_t>(num_seqs) * num_q_heads * (head_dim * 4 + 8);
        const int64_t max_parts = p.ws_bytes > 512 ? (static_cast<int64_t>(p.ws_bytes) - 512) / per_part : 1;
        p = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, dtype, true,
                      max_parts > 0 ? max_parts : 1);
        if (p.ws_bytes > workspace_bytes)
            return set_error(PKV_ERR_WORKSPACE, "decode: unaligned pools need the CUDA-core path, whose partials "
                                                "(%zu bytes) do not fit the workspace (%zu bytes)",
                             p.ws_bytes, workspace_bytes);
    }
    char *ws = static_cast<char *>(workspace);
    DecodeArgs a{out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                 num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale,
                 p.ws_bytes ? reinterpret_cast<float *>(ws) : nullptr,
                 p.ws_bytes ? reinterpret_cast<float2 *>(ws + p.o_bytes) : nullptr,
                 p.stream ? reinterpret_cast<int4 *>(ws + p.o_bytes + p.ml_bytes) : nullptr,
                 p.stream ? reinterpret_cast<int32_t *>(ws + p.o_bytes + p.ml_bytes + p.unit_bytes) : nullptr,
                 p.stream ? reinterpret_cast<uint32_t *>(ws + p.o_bytes + p.ml_bytes + p.unit_bytes + 8) : nullptr,
                 nullptr, nullptr, nullptr, nullptr, err_flag, static_cast<cudaStream_t>(stream)};
    pkv_status st;
    // The work-balanced kernel appends in its producer warp (8-byte copies);
    // every other path runs the append kernel first, in stream order.
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.codes = codes;
    const bool fused = append && fast && p.stream && aligned(new_k, 8) && aligned(new_v, 8);
    if (fused) {
        a.new_k = new_k;
        a.new_v = new_v;
    } else if (append && num_blocks > 0 && max_blocks_per_seq > 0) {
        a.new_k = new_k;
        a.new_v = new_v;
        st = launch_append(a, es);
        if (st != PKV_OK) return st;
        a.new_k = a.new_v = nullptr;
    }
    if (fast && p.stream) {
        // one work-balanced launch (and merge) per group of sequences
        const int64_t q_row = static_cast<int64_t>(num_q_heads) * head_dim * es;
        const int64_t kv_row = static_cast<int64_t>(num_kv_heads) * head_dim * es;
        for (int g = 0; g < p.groups; ++g) {
            const int b0 = g * p.group_seqs;
            DecodeArgs ag = a;
            ag.B = min(p.group_seqs, num_seqs - b0);
            ag.out = static_cast<char *>(out) + b0 * q_row;
            ag.q = static_cast<const char *>(q) + b0 * q_row;
            ag.block_tables = block_tables ? block_tables + static_cast<int64_t>(b0) * max_blocks_per_seq : nullptr;
            ag.context_lens = context_lens + b0;
            if (a.new_k) {
                ag.new_k = static_cast<const char *>(a.new_k) + b0 * kv_row;
                ag.new_v = static_cast<const char *>(a.new_v) + b0 * kv_row;
            }
            st = dtype == PKV_BF16 ? launch_stream_any<__nv_bfloat16>(ag, p) : launch_stream_any<__half>(ag, p);
            if (st != PKV_OK) return st;
        }
    } else if (fast) {
        st = dtype == PKV_BF16 ? launch_fast_any<__nv_bfloat16>(a, p) : launch_fast_any<__half>(a, p);
        if (st != PKV_OK) return st;
        st = dtype == PKV_BF16 ? launch_generic_and_combine<__nv_bfloat16>(a, p, false)
                               : launch_generic_and_combine<__half>(a, p, false);
    } else {
        switch (dtype) {
        case PKV_BF16: st = launch_generic_and_combine<__nv_bfloat16>(a, p, true); break;
        case PKV_F16: st = launch_generic_and_combine<__half>(a, p, true); break;
        default: st = launch_generic_and_combine<float>(a, p, true); break;
        }
    }
    if (st != PKV_OK) return st;
    return ok();
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_attention_decode(void *out, const void *q, const void *k_cache,
                                                 const void *v_cache, const int32_t *block_tables,
                                                 int32_t max_blocks_per_seq, const int32_t *context_lens,
                                                 int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t block_size, int32_t num_blocks,
                                                 int32_t max_context_len, float scale, pkv_dtype dtype,
                                                 void *workspace, size_t workspace_bytes,
                                                 int32_t *err_flag, void *stream) {
    return decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, dtype,
                        workspace, workspace_bytes, err_flag, stream, nullptr, nullptr);
}

extern "C" pkv_status pkv_paged_attention_decode_append(void *out, const void *q, const void *key,
                                                        const void *value, void *k_cache, void *v_cache,
                                                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                        const int32_t *context_lens, int32_t num_seqs,
                                                        int32_t num_q_heads, int32_t num_kv_heads,
                                                        int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                                        int32_t max_context_len, float scale, pkv_dtype dtype,
                                                        void *workspace, size_t workspace_bytes,
                                                        int32_t *err_flag, void *stream) {
    if (num_seqs > 0 && (!key || !value))
        return set_error(PKV_ERR_INVALID_ARG, "decode append: NULL key or value");
    return decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, dtype,
                        workspace, workspace_bytes, err_flag, stream, key, value);
}

extern "C" pkv_status pkv_paged_attention_decode_fp8(void *out, const void *q, const void *k_cache,
                                                     const void *v_cache, const float *k_scale, const float *v_scale,
                                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                     const int32_t *context_lens, int32_t num_seqs,
                                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                     int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                                     float scale, pkv_dtype dtype, void *workspace,
                                                     size_t workspace_bytes, int32_t *err_flag, void *stream) {
    if (num_seqs > 0 && (!k_scale || !v_scale))
        return set_error(PKV_ERR_INVALID_ARG, "decode fp8: NULL scales");
    if (dtype == PKV_F32) return set_error(PKV_ERR_UNSUPPORTED, "decode fp8: q/out must be fp16 or bf16");
    return decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, dtype,
                        workspace, workspace_bytes, err_flag, stream, nullptr, nullptr, k_scale, v_scale, kCodeE4M3);
}

extern "C" pkv_status pkv_paged_attention_decode_int8(void *out, const void *q, const void *k_cache,
                                                      const void *v_cache, const float *k_scale, const float *v_scale,
                                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                      const int32_t *context_lens, int32_t num_seqs,
                                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                      int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                                      float scale, pkv_dtype dtype, void *workspace,
                                                      size_t workspace_bytes, int32_t *err_flag, void *stream) {
    if (num_seqs > 0 && (!k_scale || !v_scale))
        return set_error(PKV_ERR_INVALID_ARG, "decode int8: NULL scales");
    if (dtype == PKV_F32) return set_error(PKV_ERR_UNSUPPORTED, "decode int8: q/out must be fp16 or bf16");
    return decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, dtype,
                        workspace, workspace_bytes, err_flag, stream, nullptr, nullptr, k_scale, v_scale, kCodeInt8);
}

// The fused decode step over 8-bit caches: key[b] / value[b] are encoded
// under the (block, head) scales already in k_scale / v_scale and written to
// the cache row of position context_lens[b] - 1 by the attention kernel's
// producer warp, then the attention runs over the whole context.
namespace pkv {
namespace {
pkv_status decode_append_q8(void *out, const void *q, const void *key, const void *value, void *k_cache,
                            void *v_cache, const float *k_scale, const float *v_scale, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, int32_t max_context_len, float scale, pkv_dtype dtype, void *workspace,
                            size_t workspace_bytes, int32_t *err_flag, void *stream, int32_t codes) {
    const char *fmt = codes == kCodeInt8 ? "int8" : "fp8";
    if (num_seqs > 0 && (!k_scale || !v_scale || !key || !value))
        return set_error(PKV_ERR_INVALID_ARG, "decode append %s: NULL key, value or scales", fmt);
    if (dtype == PKV_F32) return set_error(PKV_ERR_UNSUPPORTED, "decode append %s: q/out must be fp16 or bf16", fmt);
    return decode_entry(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, dtype,
                        workspace, workspace_bytes, err_flag, stream, key, value, k_scale, v_scale, codes);
}
}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_attention_decode_append_fp8(
    void *out, const void *q, const void *key, const void *value, void *k_cache, void *v_cache, const float *k_scale,
    const float *v_scale, const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, int32_t max_context_len, float scale, pkv_dtype dtype, void *workspace,
    size_t workspace_bytes, int32_t *err_flag, void *stream) {
    return decode_append_q8(out, q, key, value, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                            max_context_len, scale, dtype, workspace, workspace_bytes, err_flag, stream, kCodeE4M3);
}

extern "C" pkv_status pkv_paged_attention_decode_append_int8(
    void *out, const void *q, const void *key, const void *value, void *k_cache, void *v_cache, const float *k_scale,
    const float *v_scale, const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, int32_t max_context_len, float scale, pkv_dtype dtype, void *workspace,
    size_t workspace_bytes, int32_t *err_flag, void *stream) {
    return decode_append_q8(out, q, key, value, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                            max_context_len, scale, dtype, workspace, workspace_bytes, err_flag, stream, kCodeInt8);
}

// ----------------------------------------------------------------------------- no-allocation variant
// Decode attention for callers that cannot allocate device memory where they
// run (an engine plugin that may only use memory it was handed, a service with
// a fixed budget reserved at start-up).  The split-K scratch lives in this
// fixed region instead of a caller workspace; every GPU that loads the library
// holds it until exit.  All calls share it: nothing in it must start at zero
// (each call writes every scratch value before reading it), and calls whose GPU
// work overlaps race on it.
static __device__ __align__(256) unsigned char g_pkv_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

namespace pkv {
namespace {

// Device address of the region on the current device.  Host code cannot use
// the symbol itself (it names a host-side shadow), so the address is looked up
// with the device current, on every call: the lookup allocates nothing, and a
// fresh one stays right after a cudaDeviceReset reloads the module.
pkv_status static_workspace_address(void **addr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_pkv_static_workspace);
    if (e != cudaSuccess || !p)
        return set_error(PKV_ERR_CUDA, "static workspace: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    *addr = p;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_attention_decode_static_ws(
    void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, int32_t max_context_len,
    float scale, pkv_dtype dtype, int32_t *err_flag, void *stream) {
    // the same argument errors as the workspace variant, before the size check
    const pkv_status chk = check_decode_args(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                             context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             block_size, num_blocks, max_context_len, dtype);
    if (chk != PKV_OK) return chk;
    const size_t need = pkv_paged_attention_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                                  block_size, max_context_len, dtype);
    if (need > PKV_STATIC_WORKSPACE_BYTES)
        return set_error(PKV_ERR_WORKSPACE,
                         "decode (static workspace): these sizes need %zu bytes of scratch, more than the "
                         "library's built-in %u bytes; call pkv_paged_attention_decode with a workspace",
                         need, (unsigned)PKV_STATIC_WORKSPACE_BYTES);
    void *ws = nullptr;
    if (need > 0) {
        pkv_status st = static_workspace_address(&ws);
        if (st != PKV_OK) return st;
    }
    return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                      max_context_len, scale, dtype, ws, need > 0 ? PKV_STATIC_WORKSPACE_BYTES : 0,
                                      err_flag, stream);
}
