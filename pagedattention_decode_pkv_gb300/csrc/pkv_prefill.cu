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
// Design (fifth-generation tensor cores, FlashAttention style).  A query tile
// is 128 query rows of one KV head: 128 / G positions x the G query heads of
// the group, so every K/V byte staged for it serves all G heads.  A CTA owns
// two tiles of the same (sequence, KV head), and keys go by blocks of 128.
// Per block j:
//   * a producer warp copies K_j and V_j (the head's rows of the pages that
//     hold keys 128 j .. 128 j + 127) with TMA, in chunks of
//     gcd(block_size, 128) tokens per 64-dim half, 128-byte swizzled, into two
//     separate rings of two buffers: K_j as soon as both tiles' QKs of block
//     j - 2 have read its K buffer, V_j once their PVs of block j - 2 have
//     read its V buffer, so the K copies run ahead of the V copies and their
//     latency hides behind the PVs;
//   * an MMA warp issues, per tile, S_j = Q K_j^T (M = 128 rows, N = 128 keys,
//     eight K = 16 steps over the head dimension) into the tile's S buffer in
//     TMEM, and O += P_j V_j (N = 128 dims, K = 16 steps over the keys; P is
//     the A operand straight from TMEM, V the MN-major B operand) into the
//     tile's TMEM accumulator.  The tiles take turns: one tile's PV and next
//     QK run while the other tile's softmax works;
//   * four softmax warps per tile, one query row per thread, read the row of
//     S_j from TMEM, mask it (causal, keys of missing pages), keep the row's
//     running maximum and sum, and write P_j = exp2(S_j * scale * log2 e - m)
//     as 16-bit pairs over the S_j they read.  The next S of the tile goes into
//     that buffer right after the PV of block j that reads P_j: one thread's
//     tcgen05.mma operations run in issue order, so the MMA warp does not wait
//     for that PV.  The softmax waits for the PV of block j - 1 only when it
//     has to rescale O.
// The reference maximum m of a row moves only when the block's maximum exceeds
// it by more than 2^8 (log2 units), and then O's row is rescaled in TMEM;
// otherwise P is computed against the older m (values up to 256), which keeps
// the result the plain softmax.  The row sum adds the same rounded 16-bit P
// values the PV MMA multiplies, so the weights of the V rows sum to one (a
// single dominant key gives its V row exactly, wherever m stands).  The last
// PV's accumulator, divided by the row sum, is the output row.
// Grid (tile pairs, H_kv, B), pairs fastest: the tiles of one (sequence, KV
// head) run side by side and read its pages while they are in L2, and the tile
// index counts from the end of the sequence, so the longest tiles (most keys)
// launch first.  Every wait is bounded (PKV_ERRBIT_TIMEOUT), and the CTA waits
// for its own copies and MMAs before it frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "pkv_internal.h"
#include "pkv_pdl.cuh"
#include "pkv_tc.cuh"
#include "pkv_tma.cuh"

namespace pkv {
namespace {

constexpr int kPreRows = 128;        // query rows (position x head) per tile = TMEM lanes = MMA M
constexpr int kQHalf = kPreRows * 128;         // one 64-dim half of the Q tile [128 rows][128 dims]
constexpr int kQTileBytes = 2 * kQHalf;        // 32 KB
constexpr uint64_t kPreDeadlineNs = 2000000000ull;
constexpr float kPreLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.f;  // log2 units: P stays <= 2^8 between rescales

// acc + the low 16-bit value of w (lo) and acc2 + the high one, in f32: the
// mixed-precision adds take the 16-bit operand as it is (exact widening).
template <typename T> __device__ __forceinline__ void pair_acc(uint32_t w, float &acc, float &acc2);
template <> __device__ __forceinline__ void pair_acc<__nv_bfloat16>(uint32_t w, float &acc, float &acc2) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(acc), "+f"(acc2)
        : "r"(w));
}
template <> __device__ __forceinline__ void pair_acc<__half>(uint32_t w, float &acc, float &acc2) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(acc), "+f"(acc2)
        : "r"(w));
}

// max(a, b, c) in one instruction (three-input max; NaN operands are ignored
// as by fmaxf).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (x0, x1) * s + c per lane, both fused and rounded once (one packed f32x2 FMA);
// s2 / c2 hold the same value in both halves.
__device__ __forceinline__ void fma_x2(float x0, float x1, uint64_t s2, uint64_t c2, float &e0, float &e1) {
    asm("{\n\t.reg .b64 a, d;\n\tmov.b64 a, {%2, %3};\n\t"
        "fma.rn.f32x2 d, a, %4, %5;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(e0), "=f"(e1)
        : "f"(x0), "f"(x1), "l"(s2), "l"(c2));
}

__device__ __forceinline__ uint64_t splat2(float v) {
    const uint64_t u = __float_as_uint(v);
    return u | u << 32;
}

// Per block size (KEYS keys per block, the S MMA's N), ring depth and query
// tiles per CTA: the K/V tiles, the shared-memory layout, TMEM columns and
// mbarrier indices.  The kernel runs KEYS = 128, two buffers per ring and two
// tiles: 198 KB of shared memory (two Q tiles, K and V rings of two 32 KB
// buffers each), one CTA per SM, eight softmax warps (four per tile) sharing
// every K/V buffer.  One tile per CTA and 64-key blocks (two CTAs per SM, or
// four buffers) measured slower (launch_prefill_any).
// TMEM: tile t owns columns [t kTileCols, (t + 1) kTileCols): its S / P buffer
// (S_j in KEYS columns, then P_j in KEYS / 2 columns of 16-bit pairs written
// over the S it came from) and O at kTmemO.
template <int KEYS, int STAGES, int TILES = 1>
struct PreCfg {
    static constexpr int kNBuf = TILES == 2 && KEYS == 128 ? 1 : 2;  // S / P buffers per tile
    static constexpr uint32_t kTmemO = kNBuf * KEYS;       // O's first column within a tile
    static constexpr uint32_t kTileCols = kNBuf * KEYS + 128;
    static constexpr uint32_t kTmemCols = KEYS == 64 && TILES == 1 ? 256 : 512;  // a power of two
    static constexpr int kMinBlocks = KEYS == 64 && TILES == 1 ? 2 : 1;          // CTAs per SM
    static constexpr int kSoftWarps = 4 * TILES;           // one query row per thread
    static constexpr int kThreads = (kSoftWarps + 2) * 32;  // + producer warp + MMA warp
    static constexpr int kKvHalf = KEYS * 128;        // one 64-dim half of a K or V tile [KEYS][128 dims]
    static constexpr int kKvTileBytes = 2 * kKvHalf;
    static constexpr int kStageBytes = 2 * kKvTileBytes;  // K then V
    // shared memory
    static constexpr int kQ = 0;                                   // [TILES][2 halves][128 rows][128 B]
    static constexpr int kKV = kQ + TILES * kQTileBytes;           // stage s: K [2][KEYS][128 B], then V
    static constexpr int kKeySlots = 4;                            // blocks whose chunk key counts are kept
    static constexpr int kKeysOff = kKV + STAGES * kStageBytes;   // int32 [kKeySlots][8 chunks] valid keys
    static constexpr int kBar = kKeysOff + kKeySlots * 8 * 4;      // mbarriers, 8 bytes each
    static constexpr int kTmemSlot = kBar + 256;
    static constexpr int kBytes = kTmemSlot + 16;
    static constexpr int kAlloc = kBytes + 1024;
    // mbarrier indices; the per-buffer ones are [TILES][kNBuf] (tile-major)
    static constexpr int kBarKFull = 0;                           // [STAGES] producer: expect_tx + the K copies' bytes
    static constexpr int kBarKEmpty = kBarKFull + STAGES;         // [STAGES] MMA commit after the block's last QK
    static constexpr int kBarVFull = kBarKEmpty + STAGES;         // [STAGES] producer: expect_tx + the V copies' bytes
    static constexpr int kBarVEmpty = kBarVFull + STAGES;         // [STAGES] MMA commit after the block's last PV
    static constexpr int kBarSFull = kBarVEmpty + STAGES;         // MMA commit after S = Q K^T
    static constexpr int kBarPFull = kBarSFull + TILES * kNBuf;   // the tile's 128 softmax threads wrote P
    static constexpr int kBarODone = kBarPFull + TILES * kNBuf;   // MMA commit after O += P V
    static constexpr int kBarQFull = kBarODone + TILES * kNBuf;   // [TILES] the tile's 128 threads wrote Q
    static constexpr int kBarFinal = kBarQFull + TILES;           // MMA commit: every MMA of the CTA has completed
    static constexpr int kNumBars = kBarFinal + 1;
    static_assert(TILES == 1 || TILES == 2, "one or two query tiles per CTA");
    static_assert(kNumBars * 8 <= 256, "the mbarriers fit their shared-memory slot");
    static_assert(kKeySlots >= 2 * STAGES, "a block's key counts outlive both tiles' softmax of it");
    static_assert(TILES * kTileCols <= kTmemCols, "every tile's S buffers and O fit the TMEM allocation");
    static_assert(kAlloc * kMinBlocks <= 227 * 1024 - 1024 * (kMinBlocks - 1), "shared memory per SM");
};

template <typename T, int KEYS, int STAGES, bool POS, int TILES>
__global__ void __launch_bounds__(PreCfg<KEYS, STAGES, TILES>::kThreads, PreCfg<KEYS, STAGES, TILES>::kMinBlocks)
prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               T *__restrict__ out, const T *__restrict__ q, const int32_t *__restrict__ block_tables,
               int32_t max_blocks, const int32_t *__restrict__ starts, const int32_t *__restrict__ cu_q,
               int32_t Hq, int32_t G, int32_t bs, int32_t num_blocks, int32_t box_lg, float scale_log2,
               int32_t *__restrict__ err_flag) {
    using L = PreCfg<KEYS, STAGES, TILES>;
    constexpr int kPreKeys = KEYS, kPreStages = STAGES, kNBuf = L::kNBuf, kSoftWarps = L::kSoftWarps;
    constexpr int kKvHalf = L::kKvHalf, kKvTileBytes = L::kKvTileBytes, kStageBytes = L::kStageBytes;
    constexpr uint32_t kTmemO = L::kTmemO, kTileCols = L::kTileCols, kPreTmemCols = L::kTmemCols;
    constexpr int kBarKFull = L::kBarKFull, kBarKEmpty = L::kBarKEmpty, kBarSFull = L::kBarSFull;
    constexpr int kBarVFull = L::kBarVFull, kBarVEmpty = L::kBarVEmpty, kKeySlots = L::kKeySlots;
    static_assert(TILES == 2 && KEYS == 128, "the kernel runs two query tiles of 128-key blocks");
    constexpr int kBarPFull = L::kBarPFull, kBarODone = L::kBarODone, kBarQFull = L::kBarQFull;
    constexpr int kBarFinal = L::kBarFinal;
    using H = Half16<T>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const int b = blockIdx.z, kh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t *kv_keys = reinterpret_cast<int32_t *>(smem + L::kKeysOff);
    const uint32_t bar0 = smem_u32(smem + L::kBar);
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    const uint32_t sQ = smem_u32(smem + L::kQ), sKV = smem_u32(smem + L::kKV);
    if (warp == kSoftWarps && lane == 0) {
        for (int s = 0; s < kPreStages; ++s) {  // per K/V stage
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarKEmpty + s), 1);
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarVEmpty + s), 1);
        }
        for (int p = 0; p < TILES * kNBuf; ++p) {  // per tile and S / P buffer
            mbar_init(bar(kBarSFull + p), 1);
            mbar_init(bar(kBarPFull + p), kPreRows);
            mbar_init(bar(kBarODone + p), 1);
        }
        for (int t = 0; t < TILES; ++t) mbar_init(bar(kBarQFull + t), kPreRows);
        mbar_init(bar(kBarFinal), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    pdl_wait();
    pdl_trigger();
    const int q_begin = cu_q[b], n = cu_q[b + 1] - q_begin, start = starts[b];
    const int positions = kPreRows / G;                       // query positions per tile
    const int tiles_b = n > 0 ? (n + positions - 1) / positions : 0;
    // Tile t of the CTA is tile tiles_b - 1 - (TILES x + t) of the sequence: the
    // last tiles (most keys) launch first, and tile 0 has at least tile 1's keys.
    const int tile0 = tiles_b - 1 - static_cast<int>(blockIdx.x) * TILES;
    if ((n < 0 || tiles_b > static_cast<int>(gridDim.x) * TILES) && blockIdx.x == 0 && kh == 0 &&
        threadIdx.x == 0 && err_flag)  // cu_q decreasing, or more new tokens than max_q_len: rows left unwritten
        atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
    if (tile0 < 0) return;
    const int64_t total = static_cast<int64_t>(start) + n;
    if (start < 0 || (total + bs - 1) / bs > max_blocks) {  // a bad span: zero rows and a flag
        if (threadIdx.x == 0 && blockIdx.x == 0 && kh == 0 && err_flag) atomicOr(err_flag, PKV_ERRBIT_CONTEXT);
        const int p0 = max(tile0 - (TILES - 1), 0) * positions, p1 = min(n, (tile0 + 1) * positions);
        for (int i = threadIdx.x; i < (p1 - p0) * G * kFastHeadDim; i += blockDim.x) {
            const int pi = i / (G * kFastHeadDim), rem = i - pi * G * kFastHeadDim;
            out[(static_cast<int64_t>(q_begin + p0 + pi) * Hq + kh * G) * kFastHeadDim + rem] = from_f32<T>(0.f);
        }
        return;
    }
    // From here on the CTA holds TMEM: every path goes to the common exit below.
    if (warp == kSoftWarps + 1) tmem_alloc(smem_u32(smem + L::kTmemSlot), kPreTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    // Keys of each tile: blocks up to its last position (0 for a tile past the sequence's first).
    int nblk_t[TILES];
#pragma unroll
    for (int t = 0; t < TILES; ++t) {
        const int tt = tile0 - t;
        nblk_t[t] = tt < 0 ? 0 : (start + min(n, (tt + 1) * positions) - 1) / kPreKeys + 1;
    }
    const int nblk = nblk_t[0];
    const uint64_t deadline = global_ns() + kPreDeadlineNs;
    bool timed_out = false;

    if (warp == kSoftWarps) {
        // ------------------------------------------------------------ producer warp
        // Block j's keys come in chunks of box_rows = 2^box_lg (= gcd(block_size, 128))
        // keys: lane l < 128 / box_rows takes chunk l, whose rows are consecutive in one
        // page.  Chunks at or past the end of the span, or of a page whose id is
        // out of range, are not copied; kv_keys[stage][l] gives the consumers the
        // chunk's number of valid keys.
        const int32_t *row = block_tables + static_cast<int64_t>(b) * max_blocks;
        const int box_rows = 1 << box_lg;
        const int nch = kPreKeys / box_rows;
        const uint32_t chunk_bytes = static_cast<uint32_t>(box_rows) * 128;  // one 64-dim half of a chunk
        bool bad = false;
        int issued_k = 0, issued_v = 0;
        // Block j's K and V go to buffers j % STAGES of two separate rings: K_j
        // once both tiles' QKs of block j - STAGES have read that K buffer, V_j
        // once their PVs of block j - STAGES have read that V buffer, so the K
        // copies run a QK ahead of what one K+V stage would allow.
        auto wait_free = [&](int empty, int j) -> bool {
            int ok = 1;
            if (lane == 0 && j >= kPreStages) ok = mbar_wait(bar(empty + j % kPreStages), ((j / kPreStages) - 1) & 1, deadline);
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        for (int j = 0; j < nblk; ++j) {
            const int s = j % kPreStages;
            if (!wait_free(kBarKEmpty, j)) {
                timed_out = true;
                break;
            }
            const int key0 = j * kPreKeys + lane * box_rows;
            int id = -1, keys = 0;
            if (lane < nch && key0 < total) {  // key0 / bs < ceil(total / bs) <= max_blocks
                id = row[key0 / bs];
                if (id < 0 || id >= num_blocks) {
                    bad = true;
                } else {
                    const int64_t left = total - key0;
                    keys = left < box_rows ? static_cast<int>(left) : box_rows;
                }
            }
            if (lane < nch) kv_keys[(j % kKeySlots) * 8 + lane] = keys;
            const unsigned loaded = __ballot_sync(0xffffffffu, keys > 0);
            const uint32_t tile_bytes = static_cast<uint32_t>(__popc(loaded)) * 2u * chunk_bytes;  // K (or V) of the block
            const int slot_row = keys > 0 ? id * bs + key0 % bs : 0;
            const uint32_t kdst = sKV + static_cast<uint32_t>(s) * kStageBytes + lane * chunk_bytes;
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(bar(kBarKFull + s), tile_bytes);
            __syncwarp();
            if (keys > 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) tma_load_3d(kdst + h * kKvHalf, &tm_k, 0, slot_row, 2 * kh + h, bar(kBarKFull + s));
            }
            issued_k = j + 1;
            if (!wait_free(kBarVEmpty, j)) {
                timed_out = true;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(bar(kBarVFull + s), tile_bytes);  // after the key counts (release)
            __syncwarp();
            if (keys > 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tma_load_3d(kdst + kKvTileBytes + h * kKvHalf, &tm_v, 0, slot_row, 2 * kh + h, bar(kBarVFull + s));
            }
            issued_v = j + 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            if (bad && err_flag && kh == 0 && blockIdx.x == 0) atomicOr(err_flag, PKV_ERRBIT_BLOCK_RANGE);
            // no bulk copy may still be writing shared memory when the CTA exits
            for (int j = issued_k - kPreStages > 0 ? issued_k - kPreStages : 0; j < issued_k; ++j)
                if (!mbar_wait(bar(kBarKFull + j % kPreStages), (j / kPreStages) & 1, deadline)) timed_out = true;
            for (int j = issued_v - kPreStages > 0 ? issued_v - kPreStages : 0; j < issued_v; ++j)
                if (!mbar_wait(bar(kBarVFull + j % kPreStages), (j / kPreStages) & 1, deadline)) timed_out = true;
        }
    } else if (warp == kSoftWarps + 1) {
        // ------------------------------------------------------------ MMA warp
        if (lane == 0) {
            constexpr uint32_t kIdescS = umma_idesc_f16(kBf16, kPreRows, kPreKeys, false);
            constexpr uint32_t kIdescO = umma_idesc_f16(kBf16, kPreRows, kFastHeadDim, true);
            // S_j of tile t = Q_t K_j^T into the tile's S / P buffer once K_j has
            // landed.  The buffer's previous P (block j - 1) is read by a PV this
            // thread issued earlier: tcgen05.mma operations of one thread run in
            // issue order, so S_j may be issued without waiting for that PV.
            auto issue_qk = [&](int t, int j) -> bool {
                const int s = j % kPreStages, bj = j % kNBuf;
                bool ok = mbar_wait(bar(kBarKFull + s), (j / kPreStages) & 1, deadline);
                if (!ok) return false;
                tc_fence_after();
                const uint32_t kt = sKV + static_cast<uint32_t>(s) * kStageBytes;
                const uint32_t qt = sQ + static_cast<uint32_t>(t) * kQTileBytes;
#pragma unroll
                for (int k = 0; k < kFastHeadDim / 16; ++k) {  // 16 dims (32 bytes) per step
                    const uint32_t koff = (k & 3) * 32;
                    umma_f16(tmem + t * kTileCols + bj * kPreKeys,
                             umma_desc_sw128(qt + (k >> 2) * kQHalf + koff, 16, 1024),
                             umma_desc_sw128(kt + (k >> 2) * kKvHalf + koff, 16, 1024), kIdescS, k > 0);
                }
                umma_commit(bar(kBarSFull + t * kNBuf + bj));
                return true;
            };
            // O_t (+)= P_j V_j once the tile's softmax threads wrote P_j and V_j has landed.
            auto issue_pv = [&](int t, int j) -> bool {
                const int s = j % kPreStages, bj = j % kNBuf;
                if (!mbar_wait(bar(kBarPFull + t * kNBuf + bj), (j / kNBuf) & 1, deadline) ||
                    !mbar_wait(bar(kBarVFull + s), (j / kPreStages) & 1, deadline))
                    return false;
                tc_fence_after();
                const uint32_t vt = sKV + static_cast<uint32_t>(s) * kStageBytes + kKvTileBytes;
                const uint32_t tc = tmem + t * kTileCols;
#pragma unroll
                for (int k = 0; k < kPreKeys / 16; ++k)  // 16 keys per step: 8 P columns, two 8-row V groups
                    umma_f16_tmem_a(tc + kTmemO, tc + bj * kPreKeys + 8 * k,
                                    umma_desc_sw128(vt + k * 2048, kKvHalf, 1024), kIdescO,
                                    (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(kBarODone + t * kNBuf + bj));
                return true;
            };
            bool ok = true;
            for (int t = 0; t < TILES; ++t)
                if (ok && nblk_t[t] > 0) ok = mbar_wait(bar(kBarQFull + t), 0, deadline);
            // The tiles take turns: while one tile's softmax works on S_j, the
            // tensor core runs the other tile's PV and next QK.  A K buffer is
            // released once both tiles' QKs of its block are issued, a V buffer
            // once both PVs are (the commits arrive when those MMAs complete).
            if (ok) ok = issue_qk(0, 0);
            if (ok && nblk_t[1] > 0) ok = issue_qk(1, 0);
            if (ok) umma_commit(bar(kBarKEmpty + 0));
            for (int j = 0; ok && j < nblk; ++j) {
                ok = issue_pv(0, j);
                if (ok && j + 1 < nblk) ok = issue_qk(0, j + 1);
                if (ok && j < nblk_t[1]) ok = issue_pv(1, j);
                if (ok) umma_commit(bar(kBarVEmpty + j % kPreStages));
                if (ok && j + 1 < nblk_t[1]) ok = issue_qk(1, j + 1);
                if (ok && j + 1 < nblk) umma_commit(bar(kBarKEmpty + (j + 1) % kPreStages));
            }
            if (!ok) timed_out = true;
            umma_commit(bar(kBarFinal));  // arrives once every MMA issued above has completed
            if (!mbar_wait(bar(kBarFinal), 0, deadline)) timed_out = true;
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax warps
        // Warps 4t .. 4t + 3 serve tile t; its thread r owns query row r:
        // position index r / G, head r % G of the group.
        const int t = warp >> 2;
        const int r = threadIdx.x - t * kPreRows;
        const int my_nblk = t == 0 ? nblk_t[0] : nblk_t[TILES - 1];
        const int q0 = (tile0 - t) * positions;  // first query index of the tile
        const int pi = r / G, hd = r - pi * G;
        const bool live = my_nblk > 0 && q0 + pi < n;
        const int pos = start + q0 + pi;
        const int64_t qrow = (static_cast<int64_t>(q_begin) + q0 + pi) * Hq + kh * G + hd;
        if (my_nblk > 0) {  // Q row into shared memory (zeros past the sequence)
            const uint32_t sQt = sQ + static_cast<uint32_t>(t) * kQTileBytes;
            const int4 *src = reinterpret_cast<const int4 *>(q + qrow * kFastHeadDim);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int4 v = live ? __ldg(src + c) : make_int4(0, 0, 0, 0);
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sQt + (c >> 3) * kQHalf + r * 128 +
                                                                                (((c & 7) ^ (r & 7)) << 4)),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(bar(kBarQFull + t));
        }
        // this warp's TMEM lanes (32 (warp % 4) ..) in the tile's columns
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + t * kTileCols;
        const int bar_t = t * kNBuf;  // the tile's first S / P / O barrier
        float m_ref = -INFINITY, l_sum = 0.f;
        for (int j = 0; j < my_nblk; ++j) {
            const int s = j % kPreStages, bj = j % kNBuf;
            // S_j, then V_j: the block's key counts were written before V_j's copy
            // was armed, and tile 0 zeroes V rows of keys that were not copied.
            bool ok = mbar_wait(bar(kBarSFull + bar_t + bj), (j / kNBuf) & 1, deadline) &&
                      mbar_wait(bar(kBarVFull + s), (j / kPreStages) & 1, deadline);
            if (!__all_sync(0xffffffffu, ok)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            float x[kPreKeys];
#pragma unroll
            for (int c0 = 0; c0 < kPreKeys; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(trow + bj * kPreKeys + c0, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[c0 + i] = __uint_as_float(v[i]);
            }
            // Valid keys of each 16-key group: causal limit and the chunk's copied keys.
            int lim[kPreKeys / 16];
            {
                const int causal = live ? pos - j * kPreKeys : -1;  // keys k <= causal are visible
#pragma unroll
                for (int g = 0; g < kPreKeys / 16; ++g) {
                    const int ch = (16 * g) >> box_lg, off = 16 * g - (ch << box_lg);
                    const int copied = kv_keys[(j % kKeySlots) * 8 + ch] - off;  // valid keys of the group, from its first
                    const int c = causal - 16 * g;
                    lim[g] = min(c, min(copied, 16) - 1);      // keys 16g + i valid for i <= lim[g]
                }
            }
            bool open = true;  // every key of the block visible to this row
#pragma unroll
            for (int g = 0; g < kPreKeys / 16; ++g) open = open && lim[g] >= 15;
            // x = the scaled score (POS: the raw score, scaled inside the exponent
            // below; a positive scale keeps the maximum where it is), -inf if masked
            const float xs = POS ? 1.f : scale_log2;
            // The maximum and the sum below run as four independent chains
            // (one thread per row has no other work to hide their latency).
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (__all_sync(0xffffffffu, open)) {  // blocks below the diagonal: no mask
#pragma unroll
                for (int k = 0; k < kPreKeys; k += 2) {
                    if (!POS) {
                        x[k] *= xs;
                        x[k + 1] *= xs;
                    }
                    m4[(k >> 1) & 3] = max3f(m4[(k >> 1) & 3], x[k], x[k + 1]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kPreKeys; k += 2) {
                    x[k] = (k & 15) <= lim[k >> 4] ? x[k] * xs : -INFINITY;
                    x[k + 1] = ((k + 1) & 15) <= lim[k >> 4] ? x[k + 1] * xs : -INFINITY;
                    m4[(k >> 1) & 3] = max3f(m4[(k >> 1) & 3], x[k], x[k + 1]);
                }
            }
            float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            if (POS) mx *= scale_log2;
            float a = 1.f;
            bool resc = false;
            if (mx > m_ref + kRescaleThreshold) {  // also the row's first visible key (m_ref = -inf)
                if (m_ref != -INFINITY) {
                    a = fast_exp2(m_ref - mx);
                    resc = true;
                }
                m_ref = mx;
            }
            const float base = m_ref == -INFINITY ? 0.f : m_ref;
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            const uint64_t s2 = splat2(scale_log2), one2 = splat2(1.f), nb2 = splat2(-base);
            uint32_t pk[kPreKeys / 2];
#pragma unroll
            for (int i = 0; i < kPreKeys / 2; ++i) {
                float e0, e1;
                fma_x2(x[2 * i], x[2 * i + 1], POS ? s2 : one2, nb2, e0, e1);  // x * scale - base (POS), x - base
                pk[i] = H::pack(fast_exp2(e0), fast_exp2(e1));
                pair_acc<T>(pk[i], s4[i & 1], s4[2 + (i & 1)]);  // the rounded P the PV MMA uses: weights sum to 1
            }
            const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
            l_sum = l_sum * a + sum;
            const bool any_resc = __any_sync(0xffffffffu, resc);
            if (any_resc) {  // O changes only after the PV of block j - 1 has added to it
                ok = j == 0 || mbar_wait(bar(kBarODone + bar_t + (j - 1) % kNBuf), ((j - 1) / kNBuf) & 1, deadline);
                if (!__all_sync(0xffffffffu, ok)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
            }
            if (any_resc) {  // TMEM access is warp-wide; a = 1 leaves a row as it is
#pragma unroll
                for (int c0 = 0; c0 < kFastHeadDim; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(trow + kTmemO + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
                    tmem_st32(trow + kTmemO + c0, v);
                }
            }
            // P row over the S it came from (this thread's own columns, read
            // above): column c holds keys 2c, 2c + 1
#pragma unroll
            for (int c0 = 0; c0 < kPreKeys / 2; c0 += 32) {
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = pk[c0 + i];
                tmem_st32(trow + bj * kPreKeys + c0, v);
            }
            tmem_wait_st();
            if (t == 0 && r < kPreKeys) {  // V row of key r: zeros where nothing valid was copied (0 * NaN would poison O)
                const int g = r >> 4, ch = (16 * g) >> box_lg;
                if ((r & 15) >= kv_keys[(j % kKeySlots) * 8 + ch] - (16 * g - (ch << box_lg))) {
                    const uint32_t vrow = sKV + static_cast<uint32_t>(s) * kStageBytes + kKvTileBytes + r * 128;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + (c >> 3) * kKvHalf +
                                                                                       (c & 7) * 16),
                                     "r"(0)
                                     : "memory");
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the zeroed V rows
            tc_fence_before();
            mbar_arrive(bar(kBarPFull + bar_t + bj));
        }
        // Epilogue: O row / row sum once the last PV is done.
        bool ok = !timed_out && (my_nblk == 0 || mbar_wait(bar(kBarODone + bar_t + (my_nblk - 1) % kNBuf),
                                                            ((my_nblk - 1) / kNBuf) & 1, deadline));
        if (my_nblk == 0) {
            // a second tile past the sequence's first: nothing to write
        } else if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            T *dst = out + qrow * kFastHeadDim;
#pragma unroll
            for (int c0 = 0; c0 < kFastHeadDim; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(trow + kTmemO + c0, v);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = H::pack(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
                if (live) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<uint4 *>(dst + c0 + 8 * i) =
                            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
        } else {
            timed_out = true;
        }
    }
    // Common exit: copies landed (producer), MMAs completed (MMA warp), TMEM reads done.
    if (timed_out && err_flag) atomicOr(err_flag, PKV_ERRBIT_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kSoftWarps + 1) tmem_dealloc(tmem, kPreTmemCols);
}

template <typename T, int KEYS, int STAGES, bool POS, int TILES>
cudaError_t prefill_smem_once() {  // one flag per instantiation (they share a function type)
    static int done_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (done_dev == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(prefill_kernel<T, KEYS, STAGES, POS, TILES>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, PreCfg<KEYS, STAGES, TILES>::kAlloc);
    if (e == cudaSuccess) done_dev = dev;
    return e;
}

template <typename T, int KEYS, int STAGES, bool POS, int TILES>
pkv_status launch_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, int32_t max_blocks, const int32_t *starts,
                          const int32_t *cu_q, int32_t B, int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t bs,
                          int32_t num_blocks, float scale, int32_t *err, cudaStream_t stream) {
    // chunk = gcd(block_size, KEYS): a power of two from 16 to KEYS that divides the block
    int box_rows = KEYS;
    while (bs % box_rows) box_rows >>= 1;
    CUtensorMap mk, mv;
    const int64_t slots = static_cast<int64_t>(num_blocks) * bs;
    pkv_status st = make_kv_map_box(&mk, k_cache, Half16<T>::kTmaType, slots, Hkv, box_rows, 1);
    if (st != PKV_OK) return st;
    st = make_kv_map_box(&mv, v_cache, Half16<T>::kTmaType, slots, Hkv, box_rows, 1);
    if (st != PKV_OK) return st;
    cudaError_t e = prefill_smem_once<T, KEYS, STAGES, POS, TILES>();
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "prefill: smem attribute: %s", cudaGetErrorString(e));
    const int G = Hq / Hkv, positions = kPreRows / G;
    const int tiles = (max_q_len + positions - 1) / positions;
    using L = PreCfg<KEYS, STAGES, TILES>;
    e = launch_pdl(kPdlDecode, prefill_kernel<T, KEYS, STAGES, POS, TILES>, dim3((tiles + TILES - 1) / TILES, Hkv, B),
                   dim3(L::kThreads), L::kAlloc, stream, mk, mv, static_cast<T *>(out), static_cast<const T *>(q),
                   block_tables, max_blocks, starts, cu_q, Hq, G, bs, num_blocks, __builtin_ctz(box_rows),
                   scale * kPreLog2e, err);
    if (e != cudaSuccess) return set_error(PKV_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

// Configuration: 128-key blocks, two query tiles per CTA (eight softmax warps
// sharing each K/V stage), two stages, one CTA per SM.  Measured on GB300
// against the other configurations the kernel template admits (TFLOP/s; one
// tile of 64-key blocks with two CTAs per SM / two tiles of 64-key blocks with
// four stages / two tiles of 128-key blocks): LLaMA-shaped layer 529 / 622 /
// 722, Qwen3-shaped layer 631 / 667 / 975, 8 x 8192 513 / 612 / 741.
template <typename T>
pkv_status launch_prefill_any(void *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int32_t max_blocks, const int32_t *starts,
                              const int32_t *cu_q, int32_t B, int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t bs,
                              int32_t num_blocks, float scale, int32_t *err, cudaStream_t stream) {
    // A positive scale (the usual 1/sqrt(d)) moves into the exponent's argument.
    if (scale > 0.f)
        return launch_prefill<T, 128, 2, true, 2>(out, q, k_cache, v_cache, block_tables, max_blocks, starts, cu_q, B,
                                                  max_q_len, Hq, Hkv, bs, num_blocks, scale, err, stream);
    return launch_prefill<T, 128, 2, false, 2>(out, q, k_cache, v_cache, block_tables, max_blocks, starts, cu_q, B,
                                               max_q_len, Hq, Hkv, bs, num_blocks, scale, err, stream);
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
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
        return set_error(PKV_ERR_UNSUPPORTED, "prefill: pools, q and out must be 16-byte aligned");
    auto s = static_cast<cudaStream_t>(stream);
    pkv_status st = dtype == PKV_BF16
                        ? launch_prefill_any<__nv_bfloat16>(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                        starts, cu_q, num_seqs, max_q_len, num_q_heads, num_kv_heads,
                                                        block_size, num_blocks, scale, err_flag, s)
                        : launch_prefill_any<__half>(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, starts,
                                                 cu_q, num_seqs, max_q_len, num_q_heads, num_kv_heads, block_size,
                                                 num_blocks, scale, err_flag, s);
    if (st != PKV_OK) return st;
    return ok();
}
