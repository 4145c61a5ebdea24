// Causal varlen / chunked prefill attention over the paged KV cache.
//
// "Paged KV Cache - AI infra interview lesson": Step 3 (varlen attention and
// cu_seqlens) names prefill over sequences of different lengths and gives no
// further content; Walk the Shapes First and Step 2 give the paged layout and
// the GQA mapping.  Sequence b's new tokens occupy positions
// [starts[b], starts[b] + n_b), n_b = cu_q[b+1] - cu_q[b]; their K/V and those
// of the earlier positions are already in the cache (stored by Step 1).  Query
// i of sequence b sits at position p = starts[b] + i and attends causally:
//     out[cu_q[b] + i, h] = softmax_{t <= p}(scale * q . K[t]) . V[t],
// query head h reading KV head h / (Hq / H_kv).
//
// Design (mma.sync, FlashAttention-2 style).  A CTA owns 64 query rows of one
// KV head: 64 / G positions x the G query heads of the group, so every K/V
// byte it stages serves all G heads.  A producer warp streams 16-token K and V
// tiles of that head through a TMA -> shared-memory ring (the decode path's
// 3-D tensor map with one head per box, 128-byte swizzle).  The Q rows sit in
// shared memory (swizzled 256-byte rows), which keeps the consumers at 128
// registers and three CTAs per SM.  Four consumer warps take 16 rows each
// and, per stage, compute S = Q K^T (16 MMAs in four independent chains:
// ldmatrix of Q as A and of K as B), the online softmax on the accumulators
// (row statistics over the quad of lanes sharing a row), and O += P V (16
// MMAs: P re-used from the accumulator layout as the A operand, V through
// ldmatrix.trans).  Grid (B, H_kv, query tiles) with the tile index counted
// from the end of each sequence, so the longest tiles (most keys) launch
// first.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "pkv_pdl.cuh"
#include "pkv_tma.cuh"

namespace pkv {
namespace {

constexpr int kPreRows = 64;          // query rows (position x head) per CTA
constexpr int kPreWarps = 4;          // consumer warps, 16 rows each
constexpr int kPreStages = 6;         // K/V ring depth
constexpr int kPreTile = 2 * kStageTokens * 128;  // one head's 16 tokens of K (or V): 4 KB
constexpr uint64_t kPreDeadlineNs = 2000000000ull;
constexpr float kPreLog2e = 1.4426950408889634f;

struct PreSmem {
    static constexpr int kStageBytes = 2 * kPreTile;           // K then V
    static constexpr int kQOffset = kPreStages * kStageBytes;   // Q rows [64][256 B], chunks swizzled by row
    static constexpr int kIdOffset = kQOffset + kPreRows * 256;  // int32 block id per ring slot (-1: skipped)
    static constexpr int kBarOffset = kIdOffset + 16 * kPreStages;
    static constexpr int kBytes = kBarOffset + 16 * kPreStages;
    static constexpr int kAlloc = kBytes + 1024;
};

template <typename T>
__global__ void __launch_bounds__((kPreWarps + 1) * 32, 3)
prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               T *__restrict__ out, const T *__restrict__ q, const int32_t *__restrict__ block_tables,
               int32_t max_blocks, const int32_t *__restrict__ starts, const int32_t *__restrict__ cu_q,
               int32_t Hq, int32_t G, int32_t bs, int32_t num_blocks, float scale_log2,
               int32_t *__restrict__ err_flag) {
    using L = PreSmem;
    using H = Half16<T>;
    const int b = blockIdx.x, kh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t *ids = reinterpret_cast<int32_t *>(smem + L::kIdOffset);
    const uint32_t bar0 = smem_u32(smem + L::kBarOffset);  // full[s] = bar0 + 8s, empty[s] = bar0 + 8(STAGES+s)
    const uint32_t tiles = smem_u32(smem);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPreStages; ++i) {
            mbar_init(bar0 + 8 * i, 1);
            mbar_init(bar0 + 8 * (kPreStages + i), kPreWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();
    pdl_trigger();
    const int q_begin = cu_q[b], n = cu_q[b + 1] - q_begin, start = starts[b];
    const int positions = kPreRows / G;                       // query positions per tile
    const int tiles_b = n > 0 ? (n + positions - 1) / positions : 0;
    const int tile = tiles_b - 1 - static_cast<int>(blockIdx.z);  // the last tiles (most keys) launch first
    if ((n < 0 || tiles_b > static_cast<int>(gridDim.z)) && blockIdx.z == 0 && kh == 0 && threadIdx.x == 0 &&
        err_flag)  // cu_q decreasing, or more new tokens than max_q_len: rows left unwritten
        atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
    if (tile < 0) return;
    const int64_t total = static_cast<int64_t>(start) + n;
    if (start < 0 || (total + bs - 1) / bs > max_blocks) {  // a bad span: zero rows and a flag
        if (threadIdx.x == 0 && tile == tiles_b - 1 && kh == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
        const int p0 = tile * positions, p1 = min(n, p0 + positions);
        for (int i = threadIdx.x; i < (p1 - p0) * G * kFastHeadDim; i += blockDim.x) {
            const int pi = i / (G * kFastHeadDim), rem = i - pi * G * kFastHeadDim;
            out[(static_cast<int64_t>(q_begin + p0 + pi) * Hq + kh * G) * kFastHeadDim + rem] = from_f32<T>(0.f);
        }
        return;
    }
    __syncthreads();
    const int q0 = tile * positions;                          // first query index of the tile
    const int last_pos = start + min(n, q0 + positions) - 1;  // the tile's last position
    const int nstages = last_pos / kStageTokens + 1;
    const uint64_t deadline = global_ns() + kPreDeadlineNs;

    if (warp == kPreWarps) {
        // ------------------------------------------------------------ producer warp
        const int32_t *row = block_tables + static_cast<int64_t>(b) * max_blocks;
        bool aborted = false, bad = false;
        for (int s0 = 0; s0 < nstages && !aborted; s0 += 32) {
            const int s = s0 + lane;
            int id = -1;
            if (s < nstages) id = row[s * kStageTokens / bs];
            const int cnt = min(32, nstages - s0);
            for (int j = 0; j < cnt; ++j) {
                const int i = s0 + j, slot = i % kPreStages;
                int ok = 1;
                if (lane == 0 && i >= kPreStages)
                    ok = mbar_wait(bar0 + 8 * (kPreStages + slot), ((i / kPreStages) - 1) & 1, deadline) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    aborted = true;
                    break;
                }
                const int bid = __shfl_sync(0xffffffffu, id, j);
                if (lane == 0) {
                    const uint32_t full = bar0 + 8 * slot;
                    if (bid >= 0 && bid < num_blocks) {
                        ids[slot] = bid;
                        const int slot_row = bid * bs + (i * kStageTokens) % bs;
                        const uint32_t dst = tiles + slot * L::kStageBytes;
                        mbar_arrive_expect_tx(full, L::kStageBytes);
                        tma_load_3d(dst, &tm_k, 0, slot_row, 2 * kh, full);
                        tma_load_3d(dst + kPreTile, &tm_v, 0, slot_row, 2 * kh, full);
                    } else {
                        bad = true;
                        ids[slot] = -1;
                        mbar_arrive(full);  // nothing to load: every key of the stage is masked
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            if (aborted && err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
            if (bad && err_flag && kh == 0 && tile == tiles_b - 1) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
            // no bulk copy may still be writing shared memory when the CTA exits
            const int issued = nstages;
            for (int i = issued - kPreStages > 0 ? issued - kPreStages : 0; i < issued; ++i)
                if (!mbar_wait(bar0 + 8 * (i % kPreStages), (i / kPreStages) & 1, deadline) && err_flag)
                    atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int g = lane >> 2, t = lane & 3;
    // rows of this warp: r = 16 warp + g (and + 8) -> position index r / G, head r % G
    const int r0 = 16 * warp + g, r1 = r0 + 8;
    const int pos0 = start + q0 + r0 / G, pos1 = start + q0 + r1 / G;  // positions of the two rows
    const bool live0 = q0 + r0 / G < n, live1 = q0 + r1 / G < n;
    const int64_t qrow0 = (static_cast<int64_t>(q_begin) + q0 + r0 / G) * Hq + kh * G + r0 % G;
    const int64_t qrow1 = (static_cast<int64_t>(q_begin) + q0 + r1 / G) * Hq + kh * G + r1 % G;
    // Q rows of this warp into shared memory (zeros past the sequence): lane l
    // copies half l & 1 of row l >> 1; 16-byte chunk c of row r sits at c ^ (r & 7)
    const uint32_t qs = smem_u32(smem + L::kQOffset);
    {
        const int rw = lane >> 1, hf = lane & 1, r = 16 * warp + rw;
        const bool live = q0 + r / G < n;
        const int4 *src = reinterpret_cast<const int4 *>(
            q + ((static_cast<int64_t>(q_begin) + q0 + r / G) * Hq + kh * G + r % G) * kFastHeadDim);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            const int c = 8 * hf + c8;
            const int4 v = live ? __ldg(src + c) : make_int4(0, 0, 0, 0);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(qs + r * 256 + ((c ^ (r & 7)) << 4)),
                         "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
        }
        __syncwarp();
    }
    uint32_t q_off[8];  // A fragments by ldmatrix: rows (lane & 7) + 8 ((lane >> 3) & 1), dims 16kc + 8 (lane >> 4)
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
        const int r = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), c = 2 * kc + (lane >> 4);
        q_off[kc] = qs + r * 256 + ((c ^ (r & 7)) << 4);
    }
    // ldmatrix lane addresses inside a stage: K (B operand, non-transposed): matrix
    // m = lane >> 3 covers keys 8 (m >> 1) .. +7 and dims 16kc + 8 (m & 1) .. +7;
    // V (B operand, transposed): keys 8 (m & 1) .. +7, dims 8 (2j + (m >> 1)) .. +7.
    const int mi = lane >> 3, rr = lane & 7;
    uint32_t k_off[8], v_off[8];
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
        const int key = 8 * (mi >> 1) + rr, c16 = 2 * kc + (mi & 1);
        k_off[kc] = ((c16 >> 3) * kStageTokens + key) * 128 + (((c16 & 7) ^ (key & 7)) << 4);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int key = 8 * (mi & 1) + rr, c16 = 2 * j + (mi >> 1);
        v_off[j] = ((c16 >> 3) * kStageTokens + key) * 128 + (((c16 & 7) ^ (key & 7)) << 4);
    }
    float o[16][4];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    for (int i = 0; i < nstages; ++i) {
        const int slot = i % kPreStages;
        if (!mbar_wait(bar0 + 8 * slot, (i / kPreStages) & 1, deadline)) {
            if (lane == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
            return;
        }
        const uint32_t kt = tiles + slot * L::kStageBytes, vt = kt + kPreTile;
        const int kbase = i * kStageTokens;
        const bool skipped = ids[slot] < 0;
        if (!skipped) {
            // keys at or past the end of the sequence may hold anything, NaN
            // included: zero this stage's V rows there so that 0 * row stays 0
            const int64_t left = total - kbase;
            const int nvalid = left < kStageTokens ? static_cast<int>(left) : kStageTokens;
            if (nvalid < kStageTokens) {
                // all four consumer warps zero the same rows; each writes zeros only
                for (int idx = lane; idx < (kStageTokens - nvalid) * 16; idx += 32) {
                    const int tok = nvalid + (idx >> 4), half = (idx >> 3) & 1, chunk = idx & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                     vt + (half * kStageTokens + tok) * 128 + chunk * 16),
                                 "r"(0)
                                 : "memory");
                }
                __syncwarp();
            }
            // four independent accumulation chains (key halves x even / odd k-steps)
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kc = 0; kc < 8; kc += 2) {
                uint32_t bk[4], bk2[4], qa[4], qb[4];
                ldsm_x4(q_off[kc], qa);
                ldsm_x4(q_off[kc + 1], qb);
                ldsm_x4(kt + k_off[kc], bk);  // (keys 0-7: dims lo, hi), (keys 8-15: dims lo, hi)
                ldsm_x4(kt + k_off[kc + 1], bk2);
                H::mma(sc[0], qa, bk[0], bk[1]);
                H::mma(sc[1], qa, bk[2], bk[3]);
                H::mma(sd[0], qb, bk2[0], bk2[1]);
                H::mma(sd[1], qb, bk2[2], bk2[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
            // scores of keys kbase + 8 nt + 2t + {0, 1}, rows pos0 / pos1; causal mask
            float x[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = kbase + 8 * nt + 2 * t + e;
                    x[nt][e] = (live0 && key <= pos0) ? sc[nt][e] * scale_log2 : -INFINITY;
                    x[nt][2 + e] = (live1 && key <= pos1) ? sc[nt][2 + e] * scale_log2 : -INFINITY;
                }
            float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
            for (int sh = 1; sh < 4; sh <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = fast_exp2(m0 - base0), a1 = fast_exp2(m1 - base1);
            float p[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                p[nt][0] = fast_exp2(x[nt][0] - base0);
                p[nt][1] = fast_exp2(x[nt][1] - base0);
                p[nt][2] = fast_exp2(x[nt][2] - base1);
                p[nt][3] = fast_exp2(x[nt][3] - base1);
            }
            m0 = mn0;
            m1 = mn1;
            l0 = l0 * a0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
            l1 = l1 * a1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
            for (int dt = 0; dt < 16; ++dt) {
                o[dt][0] *= a0;
                o[dt][1] *= a0;
                o[dt][2] *= a1;
                o[dt][3] *= a1;
            }
            // P as the A operand (rows g / g+8, keys 2t.. and 8+2t..)
            uint32_t pa[4];
            pa[0] = H::pack(p[0][0], p[0][1]);
            pa[1] = H::pack(p[0][2], p[0][3]);
            pa[2] = H::pack(p[1][0], p[1][1]);
            pa[3] = H::pack(p[1][2], p[1][3]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t bv[4];
                ldsm_x4_trans(vt + v_off[j], bv);  // dims 16j .. +7: (keys 0-7, 8-15); dims 16j+8 ..: same
                H::mma(o[2 * j], pa, bv[0], bv[1]);
                H::mma(o[2 * j + 1], pa, bv[2], bv[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar0 + 8 * (kPreStages + slot));
    }
#pragma unroll
    for (int sh = 1; sh < 4; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    // C fragment: rows g / g+8, dims 8 dt + 2t, +1
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
        const int d = 8 * dt + 2 * t;
        if (live0) {
            T *dst = out + qrow0 * kFastHeadDim + d;
            dst[0] = from_f32<T>(o[dt][0] * inv0);
            dst[1] = from_f32<T>(o[dt][1] * inv0);
        }
        if (live1) {
            T *dst = out + qrow1 * kFastHeadDim + d;
            dst[0] = from_f32<T>(o[dt][2] * inv1);
            dst[1] = from_f32<T>(o[dt][3] * inv1);
        }
    }
}

template <typename K>
cudaError_t ensure_smem_once(K kernel, int bytes) {
    static int done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (done_dev == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_dev = dev;
    return e;
}

template <typename T>
pkv_status launch_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks, const int32_t *starts,
                          const int32_t *cu_q, int32_t B, int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t bs,
                          int32_t num_blocks, float scale, int32_t *err, cudaStream_t stream) {
    CUtensorMap mk, mv;
    const int64_t slots = static_cast<int64_t>(num_blocks) * bs;
    pkv_status st = make_kv_map(&mk, k_cache, Half16<T>::kTmaType, slots, Hkv, 1);
    if (st != PKV_OK) return st;
    st = make_kv_map(&mv, v_cache, Half16<T>::kTmaType, slots, Hkv, 1);
    if (st != PKV_OK) return st;
    cudaError_t e = ensure_smem_once(prefill_kernel<T>, PreSmem::kAlloc);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "prefill: smem attribute: %s", cudaGetErrorString(e));
    const int G = Hq / Hkv, positions = kPreRows / G;
    const int tiles = (max_q_len + positions - 1) / positions;
    e = launch_pdl(kPdlDecode, prefill_kernel<T>, dim3(B, Hkv, tiles), dim3((kPreWarps + 1) * 32), PreSmem::kAlloc,
                   stream, mk, mv, static_cast<T *>(out), static_cast<const T *>(q), block_tables, max_blocks, starts,
                   cu_q, Hq, G, bs, num_blocks, scale * kPreLog2e, err);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_attention_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                  const int32_t *starts, const int32_t *cu_q, int32_t num_seqs,
                                                  int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads,
                                                  int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                                  float scale, pkv_dtype dtype, int32_t *err_flag, void *stream) {
    if (dtype_bytes(dtype) == 0) return set_error(PKV_ERR_INVALID_ARG, "prefill: unknown dtype %d", (int)dtype);
    if (num_seqs < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0)
        return set_error(PKV_ERR_INVALID_ARG, "prefill: bad sizes");
    if (num_q_heads % num_kv_heads)
        return set_error(PKV_ERR_INVALID_ARG, "prefill: num_q_heads (%d) is not a multiple of num_kv_heads (%d)",
                         num_q_heads, num_kv_heads);
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return set_error(PKV_ERR_INVALID_ARG, "prefill: num_blocks * block_size >= 2^31");
    if (num_seqs > 65535 || num_kv_heads > 65535)
        return set_error(PKV_ERR_UNSUPPORTED, "prefill: more than 65535 sequences or KV heads");
    if (num_seqs == 0 || max_q_len == 0) return ok();
    const int G = num_q_heads / num_kv_heads;
    if ((dtype != PKV_F16 && dtype != PKV_BF16) || head_dim != kFastHeadDim || (G != 1 && G != 2 && G != 4 && G != 8) ||
        block_size % kStageTokens)
        return set_error(PKV_ERR_UNSUPPORTED, "prefill: needs fp16/bf16, head_dim 128, Hq/Hkv in {1, 2, 4, 8} and "
                                              "block_size a multiple of 16");
    if (!out || !q || !starts || !cu_q || !block_tables || !k_cache || !v_cache || num_blocks == 0)
        return set_error(PKV_ERR_INVALID_ARG, "prefill: NULL pointer or empty pool");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4))
        return set_error(PKV_ERR_UNSUPPORTED, "prefill: pools must be 16-byte and q/out 4-byte aligned");
    const int positions = kPreRows / G;
    if ((max_q_len + positions - 1) / positions > 65535)
        return set_error(PKV_ERR_UNSUPPORTED, "prefill: max_q_len too large for one launch");
    auto s = static_cast<cudaStream_t>(stream);
    pkv_status st = dtype == PKV_BF16
                        ? launch_prefill<__nv_bfloat16>(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                        starts, cu_q, num_seqs, max_q_len, num_q_heads, num_kv_heads,
                                                        block_size, num_blocks, scale, err_flag, s)
                        : launch_prefill<__half>(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, starts,
                                                 cu_q, num_seqs, max_q_len, num_q_heads, num_kv_heads, block_size,
                                                 num_blocks, scale, err_flag, s);
    if (st != PKV_OK) return st;
    return ok();
}
