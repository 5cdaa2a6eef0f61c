// Tensor-core (tcgen05 / TMEM / TMA) split-KV decode of the rotated-INT2 caches
// (INT2_ROT, INT2_ROT_QR) of the DeepSeek-V3 latent shape: kv_lora_rank 512, rope 64,
// block size 64, the codes expanded into fp16 operands on the fly. (The bf16 cache has
// its own kernel, mla_wide.cu.)
//
// Work decomposition. The planner cuts the concatenated 64-token tiles of all
// sequences into equal runs ("streams"); a work item is one sequence's part of
// one stream, times a tile of 128 query rows (a row is a (draft position, head)
// pair). Each stream runs on a persistent pair of CTAs that read the same KV
// tiles; CTA `half` owns latent output dims [256*half, 256*half + 256). The fp32
// latent output of 128 rows x 512 dims alone is the whole 512-column tensor
// memory of an SM, so the output is split across the pair and each CTA computes
// the scores S = Q K^T on its own (the pair shares the KV tiles through L2).
//
// Per CTA, per 64-token tile (one cache block):
//   copy    a bulk copy of the block's codes and scale/zero pairs into a raw stage,
//           expanded into an operand stage by eight dequantising warps (INT2_ROT's
//           bf16 rope key by TMA into the stage's rope block)
//   MMA     S[128 x 64]  = Q[128 x 576] . K[64 x 576]^T   (36 x M128 N64 K16, in
//           two issue groups; the first K-steps read Q from tensor memory)
//   softmax two warps per 32-row lane quarter, one per half of the tile's
//           columns: tcgen05.ld of S, causal/length mask, row max shared through
//           an mbarrier exchange, running max in log2 units with a lazy rescale
//           (only when the max grows by more than 8, so P <= 2^8), P (fp16) -> the
//           two stage blocks only QK reads (swizzled)
//   MMA     O[128 x 256] += P[128 x 64] . V[64 x 256]     (4 x M128 N256 K16,
//           issued by a warp of their own); V is the same stage read as an
//           MN-major operand
// Per work item: Q arrives by TMA (its tensor-memory part staged through the Q
// region of shared memory); the epilogue writes O / l to the bf16 partial
// buffer by TMA stores and the log2-sum-exp to the partial LSE; the combine
// kernel merges splits and applies W_UV.
//
// Tensor memory columns: O [0,256), S [256,320), Q after S.
// Roles: warp 0 = raw-block copies (+ L2 prefetch); warp 1 = TMEM owner, its lane 0
// issues the score MMAs; warps 2, 3, 12..17 = dequantisers; warps 4..11 = Q loads,
// softmax, correction and epilogue (warp w reads TMEM lanes 32*(w%4)..+31); warp 18,
// lane 0, the PV MMAs. All waits are
// bounded: a wait that gives up records FLAG_TIMEOUT and the CTA winds down
// without trapping.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>
#include <string.h>

namespace mla {
namespace tc {

// Threads per CTA: warp 0 producer, 1 score MMAs, 2, 3 and 12..17 dequantisers,
// 4..11 softmax, 18 PV MMAs (from a warp of their own, the score MMAs' issuer never
// holds them back).
constexpr int kThreads = 608;
constexpr int kPvWarp = 18;
constexpr int kTile = 64;             // tokens per tile == cache block size
constexpr int kRows = 128;            // query rows per CTA (MMA M)
constexpr int kD = 576;               // r + d_R
constexpr int kKvBlocks = 9;          // 64-dim column blocks per token row
constexpr int kStages = 2;
constexpr uint32_t kColO = 0, kColS = 256;
// Tensor-memory layout: one S buffer, Q dims 0..383 in TMEM, 384..575 in smem (the
// raw stages take the rest of the shared memory).
constexpr int kSBufs = 1, kQTmemBlocks = 6, kQSmemBlocks = 3;
constexpr int kMaxQSmemBlocks = 5;    // the Q region's size (the raw stages sit in its last two blocks)
constexpr int kSoftmaxThreads = 256;  // warps 4..11: two warps per 32-row lane quarter

constexpr uint32_t kKvBlockBytes = kTile * 128;                     // 8 KB
constexpr uint32_t kStageBytes = kKvBlocks * kKvBlockBytes;         // 72 KB
constexpr uint32_t kQBlockBytes = kRows * 128;                      // 16 KB
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffQ = kOffStage + kStages * kStageBytes;       // 144 KB
// INT2 raw stages (two): one block's codes and scale/zero pairs, copied verbatim and
// expanded into an operand stage by the dequantising warps. The bf16 rope key of
// INT2_ROT is not staged here: it is loaded by TMA straight into the operand stage's
// rope block and stays bf16 (its score K-steps take the caller's bf16 query rope dims).
// Bytes per token: codes, scale/zero pairs; INT2_ROT_QR holds the rope key as two
// more groups of codes.
template <int KIND> struct Raw {
    static constexpr bool kQR = KIND == MLA_KV_INT2_ROT_QR;
    static constexpr bool kRopeTma = KIND == MLA_KV_INT2_ROT;         // bf16 rope key by TMA
    static constexpr uint32_t kGroups = kQR ? 18 : 16;               // groups of 32 per token
    static constexpr uint32_t kCodesRow = 8 * kGroups, kSzRow = 4 * kGroups;
    static constexpr uint32_t kCodes = kTile * kCodesRow, kSz = kTile * kSzRow;
    static constexpr uint32_t kBytes = kCodes + kSz;
};
constexpr uint32_t kRawStage = Raw<MLA_KV_INT2_ROT_QR>::kBytes;      // 13.5 KB (the larger kind)
static_assert(Raw<MLA_KV_INT2_ROT>::kBytes <= kRawStage && kRawStage % 16 == 0, "raw stage sizes");
constexpr uint32_t kOffRaw = kOffQ + 3 * kQBlockBytes;              // 192 KB (INT2: after 3 Q blocks)
constexpr uint32_t kOffBar = kOffQ + kMaxQSmemBlocks * kQBlockBytes; // 224 KB
static_assert(kOffRaw + 2 * kRawStage <= kOffBar, "two INT2 raw stages must fit beside the Q blocks");
constexpr uint32_t kOffXchg = kOffBar + 512;                        // [2][128] fp32 row values
constexpr uint32_t kSmemBytes = kOffXchg + 1024 + 1024;             // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
// P (bf16 [128 rows x 64 tokens], 16 KB) of tile T is written into two column
// blocks of tile T's own stage that only QK reads (the other half's V dims),
// once QK(T) is done; PV(T) is their last reader.
__host__ __device__ constexpr uint32_t p_block(int half) { return half ? 0u : 4u; }
// rotated-INT2 cache: warps 2, 3, 12..17, two on each SM sub-partition (warp w runs
// on sub-partition w % 4), beside two softmax warps on each
constexpr int kDequantWarps = 8;
constexpr int kDequantThreads = 32 * kDequantWarps;
constexpr uint32_t kEpiBoxBytes = 32 * 128;   // epilogue box: [32 rows x 64 dims] bf16
// QK K-steps in two issue groups: [0,16) (Q from tensor memory) and [16,36). Every group boundary costs the MMA warp a warp sync and a barrier
// probe; with more, finer groups the decode ran slower.
constexpr int kQkGroups = 2;
__host__ __device__ constexpr int grp_start(int grp) {
    return grp == 0 ? 0 : grp == 1 ? 16 : 36;
}
__host__ __device__ constexpr int first_smem_group(int first_smem_step) {
    int g = 0;
    while (grp_start(g + 1) <= first_smem_step) ++g;
    return g;
}

constexpr unsigned long long kTimeoutNs = 2000000000ull;           // 2 s: a bounded-wait safety net

// Pipeline timestamps for performance analysis, compiled only with
// -DMLA_TRACE: clock64 at each hand-off of one CTA (stream MLA_TRACE_STREAM,
// half MLA_TRACE_HALF, row tile 0) for its first kTraceTiles tiles. Product builds contain none of it.
#ifdef MLA_TRACE
#ifndef MLA_TRACE_STREAM
#define MLA_TRACE_STREAM 0
#endif
#ifndef MLA_TRACE_HALF
#define MLA_TRACE_HALF 0
#endif
constexpr int kTraceTiles = 64;
__device__ long long g_trace[32][kTraceTiles];
// per CTA: start, end (globaltimer ns), items<<32 | tiles, then for items 0 and 1:
// first S seen, epilogue begin, epilogue end
__device__ unsigned long long g_cta_time[4096][9];
__device__ unsigned long long g_cta_wait[4096];   // after the grid dependency wait
#define MLA_TRACE_ITEM(slot, item)                                                               \
    do {                                                                                         \
        if ((item) < 2 && cta_id < 4096) g_cta_time[cta_id][3 + 3 * (item) + (slot)] = globaltimer(); \
    } while (0)
#define MLA_TRACE_POINT(ev, tile)                                                              \
    do {                                                                                       \
        if (blockIdx.x == MLA_TRACE_HALF && blockIdx.y == 0 && blockIdx.z == MLA_TRACE_STREAM && (tile) < kTraceTiles) \
            g_trace[ev][tile] = clock64();                                                     \
    } while (0)
#else
#define MLA_TRACE_ITEM(slot, item) \
    do {                           \
    } while (0)
#define MLA_TRACE_POINT(ev, tile) \
    do {                          \
    } while (0)
#endif
// events: 0 TMA issued, 1 stage landed (MMA), 2 QK issued, 3 S seen (softmax),
//         4 P ready (softmax), 5 PV issued, 6 PV stage released (producer saw empty),
//         7 S in registers, 8 exponentials done, 9 P about to be stored (softmax),
//         10..15 QK issue group 0..5 issued (MMA), 16 S buffer free (MMA),
//         17 first QK MMA issued, 18 about to issue it, 19 second issued, 20 tail
//         handled, 21 after the tcgen05 fence, 22 descriptors ready (MMA),
//         INT2: 24 raw block copy issued (producer), 25 raw block seen, 26 stage
//         free seen, 27 stage expanded (dequantising warp 2), 28 latent part
//         expanded (warp 2), 29 rope block landed (warp 2), 30 latent part
//         expanded (the last dequantising warp), 31 P complete (MMA)

struct Bars {
    uint64_t full[kStages];       // stage expanded (and its rope block landed)
    uint64_t empty[kStages];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full[2];
    uint64_t pv_done[2];
    uint64_t q_stage;         // a staging round of Q landed in the Q region (TMA)
    uint64_t q_smem;          // the shared-memory part of Q landed (TMA)
    uint64_t q_tmem;          // the tensor-memory part of Q is stored
    uint64_t qreg_free;       // every softmax thread is done with the Q region
    uint64_t mma_fin;
    uint64_t pv_fin;          // the PV issuer's MMAs are complete
    uint64_t xchg_full[4];    // lane quarter q: both halves of its rows wrote their value
    uint64_t xchg_read[4];    // lane quarter q: both halves read the other's value
    uint64_t raw_full[2];     // INT2: raw block landed (raw stage T % 2)
    uint64_t raw_empty[2];    // INT2: raw block read by every dequantising thread
    uint64_t rope_full[kStages];  // INT2_ROT: the bf16 rope block landed in the operand stage
    uint32_t tmem_base;
    int32_t abort_flag;
};

static_assert(sizeof(Bars) <= 512, "barriers must fit below the exchange area");

struct TcParams {
    DecodeParams p;
    int32_t row_tiles;
    uint32_t v_lbo, v_sbo;    // MN-major descriptor strides of the V operand
};

// ---------------------------------------------------------------- PTX helpers
using namespace ptx;

// Bounded wait for the phase with the given parity. On give-up it raises the
// CTA abort flag and the global timeout flag and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, Bars *bars, int32_t *status) {
    return mbar_wait_bounded(bar, parity, &bars->abort_flag, status, FLAG_TIMEOUT, kTimeoutNs);
}
__device__ __forceinline__ bool aborted(Bars *bars) { return *(volatile int32_t *)&bars->abort_flag != 0; }

// ---------------------------------------------------------------- the kernel

// Physical block of logical tile `lb` of sequence b, or -1.
__device__ __forceinline__ int block_of(const DecodeParams &p, int b, int lb) {
    if (lb >= p.max_blocks) return -1;
    const int blk = p.block_table[(size_t)b * p.max_blocks + lb];
    return (blk >= 0 && blk < p.s.num_blocks) ? blk : -1;
}

#ifndef MLA_PREFETCH_AHEAD
#define MLA_PREFETCH_AHEAD 2
#endif
constexpr int kPrefetchAhead = MLA_PREFETCH_AHEAD;   // tiles prefetched into L2 ahead of the TMA loads

// PV(Tp): O[128 x 256] += P(Tp) . V(Tp) from tile Tp's stage (4 x M128 N256 K16; P in
// the two column blocks of the other half's V dims), once the softmax has stored P;
// then commits pv_done and the stage's empty barrier. Issued by one thread.
template <int KIND>
__device__ __forceinline__ bool issue_pv(Bars *bars, uint8_t *smem, int half, const TcParams &tp, uint32_t d_o, int Tp,
                                         bool first_of_item, int32_t *status) {
    const int pb = Tp & 1;
    if (!mbar_wait(&bars->p_full[pb], (Tp >> 1) & 1, bars, status)) return false;
    MLA_TRACE_POINT(31, Tp);
    tc_fence_after();
    const int s = Tp % kStages;
    const uint64_t a0 = sdesc(smem_u32(smem + kOffStage + s * kStageBytes + p_block(half) * kKvBlockBytes), 16, 1024);
    const uint64_t b0 = sdesc(smem_u32(smem + kOffStage + s * kStageBytes) + 4 * half * kKvBlockBytes, tp.v_lbo, tp.v_sbo);
    // the operands are fp16 (the dequantised latent, P)
    constexpr uint32_t kIdPv = idesc_f16(128, 256, true);
    // descriptor start addresses advance in 16-byte units
    if (first_of_item) mma_ss_k<kIdPv, 0>(d_o, a0, b0);
    else mma_ss_k<kIdPv, 1>(d_o, a0, b0);
    mma_ss_k<kIdPv, 1>(d_o, a0 + 2, b0 + 128);
    mma_ss_k<kIdPv, 1>(d_o, a0 + 4, b0 + 256);
    mma_ss_k<kIdPv, 1>(d_o, a0 + 6, b0 + 384);
    mma_commit(&bars->pv_done[pb]);
    mma_commit(&bars->empty[s]);
    MLA_TRACE_POINT(5, Tp);
    return true;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                 const __grid_constant__ CUtensorMap o_map, const __grid_constant__ CUtensorMap rope_map,
                 const __grid_constant__ CUtensorMap qr_map, const TcParams tp) {
    using RW = Raw<KIND>;
    constexpr uint32_t kColQ = kColS + 64 * kSBufs;
    constexpr int kQRounds = (kQTmemBlocks + kQSmemBlocks - 1) / kQSmemBlocks;   // staging rounds of the TMEM part
    constexpr int kEpiBoxes = (int)((kQSmemBlocks * kQBlockBytes) / (8 * kEpiBoxBytes));   // per warp at a time
    static_assert(kEpiBoxes >= 1 && 2 % kEpiBoxes == 0, "epilogue boxes");
    // the first QK group that reads Q from shared memory
    constexpr int kFirstSmemGroup = first_smem_group(4 * kQTmemBlocks);
    const DecodeParams &p = tp.p;
    const int half = blockIdx.x;            // 0/1: which 256 latent output dims
    const int g = blockIdx.y;               // query row tile
    const int stream = blockIdx.z;          // work stream (persistent over its items)
    const int rows_seq = p.q_len * p.s.H;
#ifdef MLA_TRACE
    const unsigned cta_id = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0 && cta_id < 4096) g_cta_time[cta_id][0] = globaltimer();
#endif

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars *bars = (Bars *)(smem + kOffBar);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], kDequantThreads);
            mbar_init(&bars->empty[s], 1);
            mbar_init(&bars->rope_full[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->raw_full[i], 1);
            mbar_init(&bars->raw_empty[i], kDequantThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_free[i], kSoftmaxThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->p_full[i], kSoftmaxThreads);
            mbar_init(&bars->pv_done[i], 1);
        }
        mbar_init(&bars->q_stage, 1);
        mbar_init(&bars->q_smem, 1);
        mbar_init(&bars->q_tmem, kSoftmaxThreads);
        mbar_init(&bars->qreg_free, kSoftmaxThreads);
        mbar_init(&bars->mma_fin, 1);
        mbar_init(&bars->pv_fin, 1);
        for (int q = 0; q < 4; ++q) {          // the two softmax warps of a lane quarter
            mbar_init(&bars->xchg_full[q], 64);
            mbar_init(&bars->xchg_read[q], 64);
        }
        bars->abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    // the set-up above overlaps the planner; its schedule is read only from here on.
    // The combine may launch from here: the planner has completed, so the combine can
    // read the schedule's split ranges before its own wait.
    pdl_wait();
    pdl_trigger();
#ifdef MLA_TRACE
    if (threadIdx.x == 0 && cta_id < 4096) g_cta_wait[cta_id] = globaltimer();
#endif
    const int i0 = p.stream_start[stream], i1 = p.stream_start[stream + 1];
    if (i0 >= i1) {                          // no work for this stream (CTA-uniform)
        if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
        return;
    }

    if (warp == 0) {
        // ================================================= producer (+ L2 prefetch)
        // Lanes 0 and 1 copy the block's codes and scale/zero pairs into a raw stage
        // for the dequantising warps.
        const bool prefetcher = kPrefetchAhead > 0 && half == 0 && g == 0;
        int pi = i0, pt = 0, ahead = 0;        // L2 prefetch cursor, kPrefetchAhead tiles ahead
        auto advance_prefetch = [&]() {
            while (pi < i1 && ahead < kPrefetchAhead) {
                const WorkItem it = p.work[pi];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                if (pt >= nt) { ++pi; pt = 0; continue; }
                const int blk = block_of(p, it.b, it.t0 / kTile + pt);
                if (blk >= 0) {
                    prefetch_l2(p.codes + (size_t)blk * RW::kCodes, RW::kCodes);
                    prefetch_l2((const uint8_t *)p.scale_zero + (size_t)blk * RW::kSz, RW::kSz);
                    if (RW::kRopeTma)
                        prefetch_l2((const uint8_t *)p.rope + (size_t)blk * kKvBlockBytes, kKvBlockBytes);
                }
                ++pt;
                ++ahead;
            }
        };
        int T = 0;
        bool ok = true;
        for (int i = i0; i < i1 && ok; ++i) {
            const WorkItem it = p.work[i];
            const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
            int next_blk = block_of(p, it.b, it.t0 / kTile);     // loaded one tile ahead
            for (int t = 0; t < nt; ++t, ++T) {
                int blk = next_blk;
                if (t + 1 < nt) next_blk = block_of(p, it.b, it.t0 / kTile + t + 1);
                if (blk < 0) {            // the softmax marks the item's rows NaN
                    if (lane == 0) raise_flag(p.status, FLAG_BAD_BLOCK);
                    blk = 0;
                }
                {
                    // raw stage T % 2 is free once every dequantising thread read tile T - 2
                    const int rs = T & 1;
                    if (T >= 2 &&
                        !__all_sync(0xffffffffu, mbar_wait(&bars->raw_empty[rs], ((T - 2) >> 1) & 1, bars, p.status))) {
                        ok = false;
                        break;
                    }
                    uint8_t *raw = smem + kOffRaw + rs * kRawStage;
                    if (lane == 0) mbar_expect_tx(&bars->raw_full[rs], RW::kBytes);
                    __syncwarp();
                    if (lane == 0) bulk_load(raw, p.codes + (size_t)blk * RW::kCodes, RW::kCodes, &bars->raw_full[rs]);
                    if (lane == 1)
                        bulk_load(raw + RW::kCodes, (const uint8_t *)p.scale_zero + (size_t)blk * RW::kSz, RW::kSz,
                                  &bars->raw_full[rs]);
                    if (lane == 0) MLA_TRACE_POINT(24, T);
                }
                if (lane == 0) {                 // L2 prefetch after this tile's own loads
                    MLA_TRACE_POINT(0, T);
                    if (prefetcher && ahead > 0) --ahead;
                    if (prefetcher) advance_prefetch();
                }
            }
        }
        // drain: never leave a copy in flight into this CTA's shared memory
        for (int u = T - 2; u < T; ++u)
            if (u >= 0) mbar_drain(&bars->raw_full[u & 1], (u >> 1) & 1);
        __syncwarp();
    } else if (warp == 2 || warp == 3 || (warp >= 12 && warp < 12 + kDequantWarps - 2)) {
        // ================================================= INT2 expansion into the stage
        // value = code * scale + zero, rounded once to fp16 (the MMA operand type of
        // this cache kind), written in the 128B-swizzled layout the MMAs
        // read; the bf16 rope key (INT2_ROT) lands by TMA and stays bf16; slots past
        // the sequence end are zeroed.
        const int dw = warp < 4 ? warp - 2 : warp - 10;   // dequantising warp 0..7
        const __half2 k1024 = __float2half2_rn(1024.f);
        const int dt = 32 * dw + lane;
        int T = 0, rope_pending = -1;              // dt 0: tile whose rope copy is in flight
        bool ok = true;
        for (int i = i0; i < i1 && ok; ++i) {
            const WorkItem it = p.work[i];
            const int L = p.seq_lens[it.b];
            const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
            for (int t = 0; t < nt; ++t, ++T) {
                const int s = T % kStages, rs = T & 1;
                if (T >= kStages &&
                    !__all_sync(0xffffffffu, mbar_wait(&bars->empty[s], ((T - kStages) / kStages) & 1, bars, p.status))) {
                    ok = false;
                    break;
                }
                if (dt == 0) MLA_TRACE_POINT(26, T);
                uint8_t *stage = smem + kOffStage + s * kStageBytes;
                // the operand stage is free: its bf16 rope block comes by TMA while the
                // latent part is expanded
                if (RW::kRopeTma && dt == 0) {
                    int blk = block_of(p, it.b, it.t0 / kTile + t);
                    if (blk < 0) blk = 0;                  // the softmax marks the item's rows NaN
                    mbar_expect_tx(&bars->rope_full[s], kKvBlockBytes);
                    tma_load_2d(stage + 8 * kKvBlockBytes, &rope_map, 0, blk * kTile, &bars->rope_full[s]);
                    rope_pending = T;
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->raw_full[rs], (T >> 1) & 1, bars, p.status))) {
                    ok = false;
                    break;
                }
                if (dt == 0) MLA_TRACE_POINT(25, T);
                const int valid = min(kTile, L - (it.t0 + t * kTile));
                const uint8_t *raw = smem + kOffRaw + rs * kRawStage;
                const uint8_t *codes = raw;
                const __half *sz = (const __half *)(raw + RW::kCodes);
                // One 32-dim group (8 code bytes, one scale/zero pair) into four 16-byte
                // chunks of fp16.
                auto expand_group = [&](uint2 cb, __half2 szp, uint4 (&outc)[4]) {
                    const __half2 s2 = __half2half2(__low2half(szp)), z2 = __half2half2(__high2half(szp));
#pragma unroll
                    for (int wd = 0; wd < 2; ++wd) {
                        // 16 codes, element i at bits 2i: elements i and i + 8 sit 16 bits
                        // apart, so one mask gives the half2 (1024 + c_i, 1024 + c_{i+8})
                        // (1024 + c has the bits 0x6400 | c); subtracting 1024 gives the
                        // codes exactly, then one fused c * s + z rounded once to fp16
                        // (the operand type); byte permutes pair the values up in order.
                        const unsigned w = wd ? cb.y : cb.x;
                        uint32_t a[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const unsigned wv = ((w >> (2 * i)) & 0x00030003u) | 0x64006400u;
                            const __half2 v = __hfma2(__hsub2(*(const __half2 *)&wv, k1024), s2, z2);
                            a[i] = *(const uint32_t *)&v;
                        }
                        outc[2 * wd] = make_uint4(__byte_perm(a[0], a[1], 0x5410), __byte_perm(a[2], a[3], 0x5410),
                                                  __byte_perm(a[4], a[5], 0x5410), __byte_perm(a[6], a[7], 0x5410));
                        outc[2 * wd + 1] = make_uint4(__byte_perm(a[0], a[1], 0x7632), __byte_perm(a[2], a[3], 0x7632),
                                                      __byte_perm(a[4], a[5], 0x7632), __byte_perm(a[6], a[7], 0x7632));
                    }
                };
                // latent: a lane expands one group of one row. A warp pass covers half of
                // a row octet: lane l takes group l % 16 (distinct groups in a half-warp:
                // conflict-free code reads) of the octet's row (a + 4 (l / 16) + j) % 8,
                // a = (l / 2) % 4, pass j = 0..3 (each quarter-warp's 16-byte stores then
                // fall on eight distinct swizzled chunks: conflict-free). Each pass reads
                // its own codes (reading all four passes' first measured slower).
                static_assert(kTile / 2 == 4 * kDequantWarps, "four latent passes per dequantising warp");
                static_assert(kTile * 2 <= kDequantThreads, "one rope-group job per dequantising thread");
                const int grp = lane & 15, rho0 = ((lane >> 1) & 3) + 4 * (lane >> 4);
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int u = dw + kDequantWarps * k;
                    const int rr = 8 * (u >> 2) + ((rho0 + (u & 3)) & 7);
                    const uint2 cb = *(const uint2 *)(codes + rr * RW::kCodesRow + 8 * grp);
                    const __half2 szp = *(const __half2 *)(sz + (rr * RW::kGroups + grp) * 2);
                    uint4 outc[4];
                    if (rr < valid) {
                        expand_group(cb, szp, outc);
                    } else {                           // slots past the sequence end: zeros
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) outc[q4] = make_uint4(0, 0, 0, 0);
                    }
                    // group grp = latent chunks 4*grp .. 4*grp+3 = column block grp/2, chunks 4*(grp%2)..
                    uint8_t *blk = stage + (grp >> 1) * kKvBlockBytes;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) *(uint4 *)(blk + sw128(rr, 4 * (grp & 1) + q4)) = outc[q4];
                }
                if (RW::kQR && dt < kTile * 2) {
                    // the rope key held as codes: groups 16 and 17 of the row -> the rope block
                    const int rr = dt >> 1, gr = dt & 1;
                    const uint2 cb = *(const uint2 *)(codes + rr * RW::kCodesRow + 8 * (16 + gr));
                    const __half2 szp = *(const __half2 *)(sz + (rr * RW::kGroups + 16 + gr) * 2);
                    uint4 outc[4];
                    if (rr < valid) {
                        expand_group(cb, szp, outc);
                    } else {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) outc[q4] = make_uint4(0, 0, 0, 0);
                    }
                    uint8_t *blk = stage + 8 * kKvBlockBytes;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) *(uint4 *)(blk + sw128(rr, 4 * gr + q4)) = outc[q4];
                }
                mbar_arrive(&bars->raw_empty[rs]);    // this thread is done with the raw stage
                if (dt == 0) MLA_TRACE_POINT(28, T);
                if (dt == kDequantThreads - 32) MLA_TRACE_POINT(30, T);
                if (RW::kRopeTma) {
                    // the rope block landed as bf16, the MMA operand type of its score
                    // K-steps: only a sequence's final partial block has slots past the
                    // end to zero (stale, possibly non-finite, cache bytes)
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->rope_full[s], (T / kStages) & 1, bars, p.status))) {
                        ok = false;
                        break;
                    }
                    rope_pending = -1;
                    if (dt == 0) MLA_TRACE_POINT(29, T);
                    for (int job = dt; job < (kTile - valid) * 8; job += kDequantThreads)
                        *(uint4 *)(stage + 8 * kKvBlockBytes + sw128(valid + (job >> 3), job & 7)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async();
                mbar_arrive(&bars->full[s]);
                if (dt == 0) MLA_TRACE_POINT(27, T);
            }
        }
        // an aborted pass never leaves its rope copy in flight
        if (rope_pending >= 0) mbar_drain(&bars->rope_full[rope_pending % kStages], (rope_pending / kStages) & 1);
    } else if (warp == kPvWarp) {
        // ================================================= PV issuer: lane 0 issues
        // O += P(T) . V(T) for every tile in order as soon as the softmax has stored
        // P(T), so that the stage is released without waiting for the score MMAs of
        // the next tile to be issued; it commits its own MMAs (pv_done, empty).
        if (lane == 0) {
            const uint32_t d_o = tmem + kColO;
            bool ok = true;
            int T = 0;
            for (int i = i0; i < i1 && ok; ++i) {
                const WorkItem it = p.work[i];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                for (int t = 0; t < nt; ++t, ++T) {
                    if (!issue_pv<KIND>(bars, smem, half, tp, d_o, T, t == 0, p.status)) { ok = false; break; }
                }
            }
            mma_commit(&bars->pv_fin);
            mbar_wait(&bars->pv_fin, 0, bars, p.status);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= score MMAs: lane 0 alone runs
        // the loop (plain bounded waits, no warp-wide votes or syncs per tile)
        if (lane == 0) {
            bool ok = true;
            int T = 0;
            int item_no = 0;
            for (int i = i0; i < i1 && ok; ++i, ++item_no) {
                const WorkItem it = p.work[i];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                if (!mbar_wait(&bars->q_tmem, item_no & 1, bars, p.status)) { ok = false; break; }
                for (int t = 0; t < nt; ++t, ++T) {
                    const int s = T % kStages;
                    if (!mbar_wait(&bars->full[s], (T / kStages) & 1, bars, p.status)) { ok = false; break; }
                    MLA_TRACE_POINT(1, T);
                    // the S buffer this QK writes was read out by the softmax kSBufs tiles ago
                    if (T >= kSBufs &&
                        !mbar_wait(&bars->s_free[T % kSBufs], ((T - kSBufs) / kSBufs) & 1, bars, p.status)) {
                        ok = false;
                        break;
                    }
                    MLA_TRACE_POINT(16, T);
                    // QK(T) in kQkGroups issue groups (the dequantising warps zero a
                    // partial tile's slots past the end before they complete full[s])
                    MLA_TRACE_POINT(20, T);
                    tc_fence_after();
                    MLA_TRACE_POINT(21, T);
                    const uint64_t kd = sdesc(smem_u32(smem + kOffStage + s * kStageBytes), 16, 1024);
                    const uint64_t qd = sdesc(smem_u32(smem + kOffQ), 16, 1024);
                    const uint32_t qt = tmem + kColQ;
                    const uint32_t d_s = tmem + kColS + 64 * (T % kSBufs);
                    MLA_TRACE_POINT(22, T);
                    constexpr uint32_t kIdQk = idesc_f16(128, 64, false);
#pragma unroll
                    for (int grp = 0; grp < kQkGroups; ++grp) {
                        // the item's first tile: its shared-memory Q part may still be landing
                        if (grp == kFirstSmemGroup && t == 0 && !mbar_wait(&bars->q_smem, item_no & 1, bars, p.status)) {
                            ok = false;
                            break;
                        }
                        // K-step j: column block j/4, 32-byte step j%4 inside the swizzle
                        // atom; descriptor start addresses advance in 16-byte units.
#pragma unroll
                        for (int j = grp_start(grp); j < grp_start(grp + 1); ++j) {
                            const uint64_t bd = kd + (uint64_t)(((j >> 2) * kKvBlockBytes + 32 * (j & 3)) >> 4);
                            if (j == 0) {
                                MLA_TRACE_POINT(18, T);
                                mma_ts_k<kIdQk, 0>(d_s, qt, bd);
                                MLA_TRACE_POINT(17, T);
                            } else if (j == 1) {
                                mma_ts_k<kIdQk, 1>(d_s, qt + 8 * j, bd);
                                MLA_TRACE_POINT(19, T);
                            } else if (j < 4 * kQTmemBlocks) {
                                mma_ts_k<kIdQk, 1>(d_s, qt + 8 * j, bd);
                            } else if (RW::kRopeTma && j >= 4 * (kKvBlocks - 1)) {
                                // INT2_ROT: the rope block is bf16 on both sides (the key as
                                // cached, the caller's query); the same fp32 accumulator
                                constexpr uint32_t kIdRope = idesc_bf16(128, 64, false);
                                mma_ss_k<kIdRope, 1>(
                                    d_s, qd + (uint64_t)((((j >> 2) - kQTmemBlocks) * kQBlockBytes + 32 * (j & 3)) >> 4), bd);
                            } else {
                                mma_ss_k<kIdQk, 1>(
                                    d_s, qd + (uint64_t)((((j >> 2) - kQTmemBlocks) * kQBlockBytes + 32 * (j & 3)) >> 4), bd);
                            }
                        }
                        MLA_TRACE_POINT(10 + grp, T);
                    }
                    if (!ok) break;
                    mma_commit(&bars->s_full[T % kSBufs]);
                    MLA_TRACE_POINT(2, T);
                }
            }
            mma_commit(&bars->mma_fin);
            mbar_wait(&bars->mma_fin, 0, bars, p.status);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ================================================= Q loads, softmax, epilogue
        // Warps 4..11: warp w owns rows 32*(w%4)..+31 (its TMEM lane quarter) and
        // half hs = (w-4)/4 of each row: score columns 32*hs..+31, output columns
        // 128*hs..+127. The two halves of a row agree on the running max through
        // shared memory once per tile. Every branch around tcgen05.ld / tcgen05.st
        // is warp-uniform: those instructions are warp-collective (.sync.aligned).
        //
        // The Q region of shared memory serves three uses in turn: staging the
        // tensor-memory part of an item's Q (TMA in, tcgen05.st out), the
        // epilogue's output boxes (written here, TMA-stored out) and the
        // shared-memory part of Q that the QK MMAs read. qreg_free completes once
        // every softmax thread is done with a staging or epilogue use; the TMA
        // issuer (warp 4 lane 0) waits for it before loading into the region.
        const int wq = warp & 3;
        const int hs = (warp - 4) >> 2;
        const int row = 32 * wq + lane;
        const int row_seq = g * kRows + row;
        const bool row_valid = row_seq < rows_seq;
        const bool issuer = warp == 4 && lane == 0;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16);
        float *xchg = (float *)(smem + kOffXchg);       // [2][128]
        bool ok = true;
        int T = 0;
        int nx = 0;                                     // exchanges done
        int uses = 0;                                   // qreg_free phases this thread arrived on
        int nstage = 0;                                 // q_stage phases consumed
        // Swap one value per row with the other half of the row (bounded waits).
        auto exchange = [&](float v, float &other) -> bool {
            if (nx > 0 && !mbar_wait(&bars->xchg_read[wq], (nx - 1) & 1, bars, p.status)) return false;
            xchg[hs * 128 + row] = v;
            mbar_arrive(&bars->xchg_full[wq]);
            if (!mbar_wait(&bars->xchg_full[wq], nx & 1, bars, p.status)) return false;
            other = xchg[(hs ^ 1) * 128 + row];
            mbar_arrive(&bars->xchg_read[wq]);
            ++nx;
            return true;
        };
        // TMA of Q part `round` of work item `item` into the Q region (issuer
        // only). Rounds 0..kQRounds-1 stage the tensor-memory part, kQRounds
        // loads the shared-memory part that the MMAs read.
        auto issue_q = [&](int item, int round) -> bool {
            if (!issuer) return true;
            if (uses > 0 && !mbar_wait(&bars->qreg_free, (uses - 1) & 1, bars, p.status)) return false;
            const int qrow = p.work[item].b * rows_seq + g * kRows;
            int first, n;
            uint64_t *bar;
            if (round < kQRounds) {
                first = round * kQSmemBlocks;
                n = min(kQSmemBlocks, kQTmemBlocks - first);
                bar = &bars->q_stage;
            } else {
                first = kQTmemBlocks;
                n = kQSmemBlocks;
                bar = &bars->q_smem;
            }
            mbar_expect_tx(bar, (uint32_t)n * kQBlockBytes);
            for (int k = 0; k < n; ++k) {
                // INT2_ROT: the rope block (8) straight from the caller's bf16 query
                const bool rope_bf16 = RW::kRopeTma && first + k == kKvBlocks - 1;
                tma_load_2d(smem + kOffQ + k * kQBlockBytes, rope_bf16 ? &qr_map : &q_map, 64 * (first + k), qrow, bar);
            }
            return true;
        };
        // Staged round -> tensor memory: each thread moves its row's 64-dim
        // blocks (those with block index % 2 == hs) with tcgen05.st.
        auto stage_q = [&](int round) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_stage, nstage & 1, bars, p.status))) return false;
            ++nstage;
            const int first = round * kQSmemBlocks;
            const int n = min(kQSmemBlocks, kQTmemBlocks - first);
#pragma unroll 1
            for (int k = hs; k < n; k += 2) {
                uint32_t v[32];
                const uint8_t *blk = smem + kOffQ + k * kQBlockBytes;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 u = *(const uint4 *)(blk + sw128(row, ch));
                    v[4 * ch + 0] = u.x;
                    v[4 * ch + 1] = u.y;
                    v[4 * ch + 2] = u.z;
                    v[4 * ch + 3] = u.w;
                }
                TMEM_ST32(lane_addr + kColQ + 32 * (first + k), v);
            }
            mbar_arrive(&bars->qreg_free);
            ++uses;
            return true;
        };
        // All staging rounds of `item` (round 0 already issued); then the
        // tensor-memory part of Q is complete for the MMA warp.
        auto load_q_tmem = [&](int item) -> bool {
            for (int r = 0; r < kQRounds; ++r) {
                if (r > 0 && !__all_sync(0xffffffffu, issue_q(item, r))) return false;
                if (!stage_q(r)) return false;
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->q_tmem);
            return true;
        };
        // ---- Q of the first item
        ok = __all_sync(0xffffffffu, issue_q(i0, 0));
        ok = ok && load_q_tmem(i0);
        ok = ok && __all_sync(0xffffffffu, issue_q(i0, kQRounds));
        for (int i = i0; i < i1 && ok; ++i) {
            const WorkItem it = p.work[i];
            const int L = p.seq_lens[it.b];
            const int t0 = it.t0, t1 = it.t1;
            const int nt = (t1 - t0 + kTile - 1) / kTile;
            const int last_vis = L - p.q_len + (row_valid ? row_seq / p.s.H : 0);
            float m_used = -CUDART_INF_F, l = 0.f;       // l: this half's share of the row sum
            bool bad_item = false;     // a block id of this item is out of range
            for (int t = 0; t < nt && ok; ++t, ++T) {
                bad_item |= block_of(p, it.b, t0 / kTile + t) < 0;
                const int sb = T % kSBufs;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (T / kSBufs) & 1, bars, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (row == 0 && hs == 0) MLA_TRACE_POINT(3, T);
                if (row == 0 && hs == 0 && t == 0) MLA_TRACE_ITEM(0, i - i0);
                uint32_t sv[32];
                TMEM_LD32(lane_addr + kColS + 64 * sb + 32 * hs, sv);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars->s_free[sb]);
                if (row == 0 && hs == 0) MLA_TRACE_POINT(7, T);

                const int tile_start = t0 + t * kTile + 32 * hs;
                // tokens j < n_vis of this half-tile are visible to this row
                const int n_vis = row_valid ? max(0, min(t1, last_vis + 1) - tile_start) : 0;
                // Scores stay unscaled where the scale is positive: the row max then
                // commutes with the scaling (rounding is monotonic) and each exponent
                // argument is a single fma, s * scale - max. Hidden slots become -inf
                // (only partial tiles pay for the mask).
                const bool pos_scale = p.scale_log2 > 0.f;
                const float cs = pos_scale ? p.scale_log2 : 1.f;
                if (!pos_scale || __any_sync(0xffffffffu, n_vis < 32)) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float v = pos_scale ? __uint_as_float(sv[j]) : __uint_as_float(sv[j]) * p.scale_log2;
                        sv[j] = __float_as_uint(j < n_vis ? v : -CUDART_INF_F);
                    }
                }
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(sv[j]));
                mx *= cs;
                // the row's max over both halves
                {
                    float other = -CUDART_INF_F;
                    if (!__all_sync(0xffffffffu, exchange(mx, other))) { ok = false; break; }
                    mx = fmaxf(mx, other);
                }
                float alpha = 1.f;
                bool rescale = false;
                const float m_new = fmaxf(m_used, mx);
                if (m_new > m_used + 8.f) {
                    alpha = exp2f(m_used - m_new);        // 0 when nothing was accumulated yet
                    m_used = m_new;
                    rescale = t > 0;
                }
                // minus the exponent base: -(running max), or -inf for a row with
                // nothing visible yet (every argument is then -inf and P = 0)
                const float nmb = m_used == -CUDART_INF_F ? -CUDART_INF_F : -m_used;
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float a = ex2(fmaf(__uint_as_float(sv[2 * j]), cs, nmb));
                    const float c = ex2(fmaf(__uint_as_float(sv[2 * j + 1]), cs, nmb));
                    const __half2 h = __floats2half2_rn(a, c);     // P: fp16, the PV operand type
                    pk[j] = *(const uint32_t *)&h;
                    sum0 += a;             // fp32 row sum: the LSE does not see the rounding of P
                    sum1 += c;
                }
                if (row == 0 && hs == 0) MLA_TRACE_POINT(8, T);
                l = l * alpha + (sum0 + sum1);
                const int pb = T & 1;
                if (row == 0 && hs == 0) MLA_TRACE_POINT(9, T);
                // Rows decide to rescale on their own; the warp corrects its O columns
                // together (alpha = 1 for rows that keep their max).
                if (__any_sync(0xffffffffu, rescale)) {
                    // O *= alpha once PV(T-1) has landed; PV(T) waits for p_full below
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&bars->pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, bars, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 4 * hs; c < 4 * hs + 4; ++c) {
                        uint32_t ov[32];
                        TMEM_LD32(lane_addr + kColO + 32 * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
                        TMEM_ST32(lane_addr + kColO + 32 * c, ov);
                    }
                    tmem_wait_st();
                }
                uint8_t *pbuf = smem + kOffStage + (T % kStages) * kStageBytes + p_block(half) * kKvBlockBytes;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *(uint4 *)(pbuf + sw128(row, 4 * hs + ch)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&bars->p_full[pb]);
                if (row == 0 && hs == 0) MLA_TRACE_POINT(4, T);
            }
            // ---- end of this item. The Q region is free (the item's last QK has
            // completed): stage the next item's tensor-memory Q while the last PV
            // runs, then write this item's output through the region, then load
            // the next item's shared-memory Q part.
            const bool have_next = i + 1 < i1;
            if (ok && have_next) ok = __all_sync(0xffffffffu, issue_q(i + 1, 0));
            if (row == 0 && hs == 0) MLA_TRACE_ITEM(1, i - i0);
            if (ok && nt > 0) {
                const int tl = T - 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->pv_done[tl & 1], (tl >> 1) & 1, bars, p.status));
            }
            // the row sum over both halves
            float l_other = 0.f;
            if (ok) ok = __all_sync(0xffffffffu, exchange(l, l_other));
            const float l_row = l + l_other;
            tc_fence_after();
            // O (fp32, this half's 256 latent dims) leaves tensor memory before the
            // next item's staged Q enters it: both use the same lane quarter.
            if (ok && have_next) ok = load_q_tmem(i + 1);
            if (ok && have_next)        // every thread has read its staged Q out of the region
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->qreg_free, (uses - 1) & 1, bars, p.status));
            const bool bad = aborted(bars) || !ok || bad_item;
            // Epilogue: O / l -> partial slot i, rounded to bf16 (the combine rounds the
            // merged rows to a bf16 MMA operand as well). Each warp writes [32 rows x 64
            // dims] boxes (128B-swizzled) into the region, kEpiBoxes at a time, and
            // stores each with one TMA copy; rows past the sequence's rows are clipped
            // by the tensor map.
            if (ok) {
                const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                // the partials are read back by the combine right after this kernel:
                // keep them in L2 over the KV stream, which is read once
                const uint64_t keep = l2_policy_evict_last();
                uint8_t *boxes = smem + kOffQ + (warp - 4) * kEpiBoxes * kEpiBoxBytes;
                const int y = g * kRows + 32 * wq;
                const bool store = y < rows_seq;                 // warp-uniform
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    const int bi = c % kEpiBoxes;
                    if (bi == 0 && c > 0) {                      // the previous boxes were read
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
                    }
                    uint8_t *box = boxes + bi * kEpiBoxBytes;
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {             // 32 of the box's 64 dims at a time
                        uint32_t ov[32];
                        TMEM_LD32(lane_addr + kColO + 128 * hs + 64 * c + 32 * hh, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {            // 16-byte chunk 4 hh + q: 8 dims
                            uint32_t pk[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                    __uint_as_float(ov[8 * q + 2 * e]) * inv, __uint_as_float(ov[8 * q + 2 * e + 1]) * inv);
                                pk[e] = *(const uint32_t *)&h2;
                            }
                            *(uint4 *)(box + sw128(lane, 4 * hh + q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0 && store) {
                        tma_store_3d_hint(&o_map, box, 256 * half + 128 * hs + 64 * c, y, i, keep);
                        bulk_commit();
                    }
                }
                if (lane == 0) bulk_wait_read();
                __syncwarp();
            }
            mbar_arrive(&bars->qreg_free);
            ++uses;
            if (row_valid && half == 0 && hs == 0)
                p.part_lse[(size_t)i * rows_seq + row_seq] =
                    bad ? CUDART_NAN_F : (l_row > 0.f ? m_used + log2f(l_row) : -CUDART_INF_F);
            tc_fence_before();     // O reads complete before the next item's first PV
            if (ok && have_next) ok = __all_sync(0xffffffffu, issue_q(i + 1, kQRounds));
            if (row == 0 && hs == 0) MLA_TRACE_ITEM(2, i - i0);
        }
        if (lane == 0) bulk_wait_all();   // this warp's output stores have landed
    }
    tc_fence_before();
    __syncthreads();
#ifdef MLA_TRACE
    if (threadIdx.x == 0 && cta_id < 4096) {
        g_cta_time[cta_id][1] = globaltimer();
        int nt = 0;
        for (int i = i0; i < i1; ++i) nt += (p.work[i].t1 - p.work[i].t0 + kTile - 1) / kTile;
        g_cta_time[cta_id][2] = ((unsigned long long)(i1 - i0) << 32) | (unsigned)nt;
    }
#endif
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

// 2-D map over the first `cols` columns (576 by default) of a row-major
// [rows, row_elems] matrix of 16-bit elements (bf16 or fp16), 128-byte swizzled
// boxes of [box_rows, 64]. Rows past the end read as zero.
static bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows,
                     CUtensorMapDataType dtype, uint64_t row_elems = kD, uint64_t cols = kD) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D bf16 map over the partial outputs [slots, rows_seq, r], boxes of
// [32 rows x 64 dims] with the 128-byte swizzle (stores clip rows >= rows_seq).
static bool make_out_map(CUtensorMap *map, void *base, int r, int rows_seq, int slots) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)r, (cuuint64_t)rows_seq, (cuuint64_t)slots};
    cuuint64_t strides[2] = {(cuuint64_t)r * 2, (cuuint64_t)rows_seq * r * 2};
    cuuint32_t box[3] = {64, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

}  // namespace tc

bool tc_shape_supported(const ShapeArgs &s) {
    if (s.r != 512 || s.dR != 64 || s.bs != tc::kTile) return false;
    return s.kind == MLA_KV_BF16 || ((s.kind == MLA_KV_INT2_ROT || s.kind == MLA_KV_INT2_ROT_QR) && s.gs == 32);
}

cudaError_t launch_decode_tc(const DecodeParams &p, int32_t max_work, cudaStream_t st) {
    // the bf16 cache: two cache blocks per score MMA (mla_wide.cu)
    if (p.s.kind == MLA_KV_BF16) return launch_decode_wide(p, max_work, st);
    tc::TcParams tp;
    tp.p = p;
    tp.row_tiles = (p.q_len * p.s.H + tc::kRows - 1) / tc::kRows;
    // MN-major V operand: 64-dim atoms 8 KB apart, 8-token groups 1 KB apart.
    tp.v_lbo = tc::kKvBlockBytes;
    tp.v_sbo = 1024;
    CUtensorMap q_map, o_map, rope_map;
    memset(&rope_map, 0, sizeof rope_map);
    // INT2_ROT: the caller's bf16 query, read for its rope block only
    CUtensorMap qr_map;
    memset(&qr_map, 0, sizeof qr_map);
    if (p.s.kind == MLA_KV_INT2_ROT &&
        !tc::make_map(&qr_map, p.q_rope, (uint64_t)p.B * p.q_len * p.s.H, tc::kRows, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return cudaErrorInvalidValue;
    // INT2_ROT: the bf16 rope keys [num_blocks * block_size, d_R], one 64-row box a tile
    if (p.s.kind == MLA_KV_INT2_ROT &&
        !tc::make_map(&rope_map, p.rope, (uint64_t)p.s.num_blocks * p.s.bs, tc::kTile, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      (uint64_t)p.s.dR, (uint64_t)p.s.dR))
        return cudaErrorInvalidValue;
    // the fp16 rotated query
    const int rows_seq = p.q_len * p.s.H;
    if (!tc::make_map(&q_map, p.q, (uint64_t)p.B * rows_seq, tc::kRows, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
        return cudaErrorInvalidValue;
    if (!tc::make_out_map(&o_map, p.part_o, p.s.r, rows_seq, max_work)) return cudaErrorInvalidValue;
    auto kern = p.s.kind == MLA_KV_INT2_ROT_QR ? tc::decode_tc_kernel<MLA_KV_INT2_ROT_QR>
                                              : tc::decode_tc_kernel<MLA_KV_INT2_ROT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(2, tp.row_tiles, p.streams);
    return launch_pdl(kern, grid, dim3(tc::kThreads), tc::kSmemBytes, st, q_map, o_map, rope_map, qr_map, tp);
}

}  // namespace mla

#ifdef MLA_TRACE
extern "C" int mla_trace_read(long long *host, int n) {
    return (int)cudaMemcpyFromSymbol(host, mla::tc::g_trace, sizeof(long long) * (size_t)n);   // [32][64]
}
extern "C" int mla_trace_cta_wait(unsigned long long *host, int n) {
    return (int)cudaMemcpyFromSymbol(host, mla::tc::g_cta_wait, sizeof(unsigned long long) * (size_t)n);
}
extern "C" int mla_trace_cta(unsigned long long *host, int n) {
    return (int)cudaMemcpyFromSymbol(host, mla::tc::g_cta_time, sizeof(unsigned long long) * 9 * (size_t)n);
}
#endif

