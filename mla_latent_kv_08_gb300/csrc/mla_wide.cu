// Tensor-core (tcgen05 / TMEM / TMA) split-KV decode of the bf16 latent cache of the
// DeepSeek-V3 shape (kv_lora_rank 512, rope 64, block size 64) that scores two cache
// blocks per MMA: each score MMA is M128 N128 K16 over 128 tokens.
//
// Why. A score MMA M128 K16 costs about the same issue time for N = 64 as for N = 128,
// so scoring one 64-token block per MMA runs the tensor pipe at half rate on the largest
// MMA work of the decode (36 K-steps over the 576 dims for every block). Here a step is
// two consecutive blocks of one sequence, laid out so that each 64-dim column block of
// the step is one [128 tokens x 128 B] K-major operand: tile 0 in rows 0..63, tile 1 in
// rows 64..127. The step's 144 KB and the query's shared-memory part (80 KB) fill shared
// memory, so there is one step buffer, released in two parts: the five column blocks
// only the scores read (the other half's latent dims and the rope key) once the score
// MMAs over them complete, the four blocks of this CTA's own latent dims once PV is done.
// P is stored by the softmax into tensor memory over the scores it replaces and is read
// from there by PV as the A operand, so no shared memory holds it.
//
// As in the single-block kernel, CTA `half` of a pair owns latent output dims
// [256*half, 256*half + 256) and the pair shares the KV tiles through L2; each CTA
// computes the scores on its own.
//
// Per CTA, per step of 128 tokens:
//   TMA     the 5 score-only column blocks of both tiles (10 boxes [64 tokens x 64 dims],
//           128B-swizzled), then the 4 own column blocks (8 boxes); a missing second tile
//           (an odd block count) is read past the end of the cache, which fills zeros
//   MMA     S[128 x 128] = Q . K^T: 20 K-steps with Q's shared-memory part over the
//           score-only blocks, then 16 with Q's tensor-memory part over the own blocks
//   softmax two warps per 32-row lane quarter, one per 64-token half: tcgen05.ld of S,
//           causal/length mask, row max shared through shared memory, running max in
//           log2 units raised lazily (only when it grows by more than 8), P in bf16 by
//           tcgen05.st into tensor memory over S
//   MMA     O[128 x 256] += P[128 x 128] . V[128 x 256]: 8 x M128 N256 K16, A = P in
//           tensor memory, B = the own column blocks read as an MN-major operand
// Per work item (one sequence's run of blocks on one stream): Q arrives by TMA, its
// tensor-memory part staged through the Q region of shared memory; the epilogue writes
// O / l to the bf16 partial buffer by TMA stores and the log2-sum-exp to the partial LSE;
// the combine kernel merges splits and applies W_UV.
//
// Tensor memory: O [0,256), S / P [256,384), Q's own latent dims [384,512).
// Roles: warp 0 = TMA producer (+ L2 prefetch, + zeroing of a partial tile's own rows
// past the sequence end); warp 1 = TMEM owner, lane 0 issues every MMA; warps 4..11 = Q
// loads, softmax and epilogue (warp w reads TMEM lanes 32*(w%4)..+31). Every wait is
// bounded (2 s); a wait that gives up records FLAG_TIMEOUT and the CTA winds down
// without trapping.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>
#include <string.h>

namespace mla {
namespace wide {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;                  // warps 4..11
constexpr int kTile = 64;                             // tokens per cache block
constexpr int kStep = 2 * kTile;                      // tokens per step (MMA N of the scores)
constexpr int kRows = 128;                            // query rows per CTA (MMA M)
constexpr int kD = 576;                               // r + d_R
constexpr int kBlocks = 9;                            // 64-dim column blocks per token row
constexpr uint32_t kBox = kTile * 128;                // [64 tokens x 64 dims] bf16: 8 KB
constexpr uint32_t kCol = kStep * 128;                // one column block of a step: 16 KB
constexpr uint32_t kQBlock = kRows * 128;             // [128 rows x 64 dims] bf16: 16 KB
constexpr int kQTmemBlocks = 4;                       // Q's own latent dims
constexpr int kQSmemBlocks = 5;                       // Q's score-only dims
constexpr uint32_t kOffBuf = 0;
constexpr uint32_t kOffQ = kOffBuf + kBlocks * kCol;          // 144 KB
constexpr uint32_t kOffBar = kOffQ + kQSmemBlocks * kQBlock;   // 224 KB
constexpr uint32_t kOffXchg = kOffBar + 512;                   // [2][128] fp32 row values
constexpr uint32_t kSmemBytes = kOffXchg + 1024 + 1024;        // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 384;
constexpr uint32_t kEpiBoxBytes = 32 * 128;           // epilogue box: [32 rows x 64 dims] bf16
constexpr int kEpiBoxes = (int)((kQSmemBlocks * kQBlock) / (8 * kEpiBoxBytes));   // per warp at a time
static_assert(kEpiBoxes >= 1 && 2 % kEpiBoxes == 0, "epilogue boxes");
constexpr unsigned long long kTimeoutNs = 2000000000ull;       // 2 s bounded-wait safety net
#ifndef MLA_WIDE_PREFETCH_AHEAD
#define MLA_WIDE_PREFETCH_AHEAD 4
#endif
constexpr int kPrefetchAhead = MLA_WIDE_PREFETCH_AHEAD;       // blocks prefetched into L2 ahead

// Column block of the step buffer that holds dims [64c, 64c + 64): own blocks are the
// latent blocks 4*half .. 4*half + 3; the five score-only blocks are the other half's
// latent blocks and the rope block (index 8).
__device__ __forceinline__ int score_only_block(int half, int k) { return k < 4 ? 4 * (1 - half) + k : 8; }

// Pipeline timestamps for performance analysis, compiled only with -DMLA_TRACE: clock64
// at each hand-off of one CTA (stream MLA_TRACE_STREAM, half MLA_TRACE_HALF, row tile 0)
// for its first kTraceSteps steps. Product builds contain none of it.
#ifdef MLA_TRACE
#ifndef MLA_TRACE_STREAM
#define MLA_TRACE_STREAM 0
#endif
#ifndef MLA_TRACE_HALF
#define MLA_TRACE_HALF 0
#endif
constexpr int kTraceSteps = 64;
__device__ long long g_wtrace[12][kTraceSteps];
// per CTA (globaltimer): entry, after the grid dependency wait, end
__device__ unsigned long long g_wcta[2048][3];
#define WTRACE(ev, step)                                                                                          \
    do {                                                                                                          \
        if (blockIdx.x == MLA_TRACE_HALF && blockIdx.y == 0 && blockIdx.z == MLA_TRACE_STREAM && (step) < kTraceSteps) \
            g_wtrace[ev][step] = clock64();                                                                       \
    } while (0)
#else
#define WTRACE(ev, step) \
    do {                 \
    } while (0)
#endif
// events: 0 score-only boxes issued, 1 own boxes issued (producer), 2 score-only blocks
// landed, 3 part 1 issued, 4 own blocks landed, 5 QK committed, 6 P seen, 7 PV issued
// (MMA), 8 S seen, 9 row max agreed, 10 P stored (softmax), 11 entry

struct Bars {
    uint64_t full_a;          // the step's score-only blocks landed
    uint64_t full_v;          // the step's own blocks landed
    uint64_t empty_a;         // the score MMAs over the score-only blocks completed
    uint64_t empty_v;         // PV of the step completed
    uint64_t tail_done;       // the producer zeroed a partial tile's own rows past the end
    uint64_t s_full;
    uint64_t p_full;
    uint64_t pv_done;
    uint64_t q_stage;         // the staged tensor-memory part of Q landed in the Q region
    uint64_t q_smem;          // Q's shared-memory part landed in the Q region
    uint64_t q_tmem;          // the tensor-memory part of Q is stored
    uint64_t qreg_free;       // every softmax thread is done with the Q region
    uint64_t mma_fin;
    uint64_t xchg_full[4];    // lane quarter q: both halves of its rows wrote their value
    uint64_t xchg_read[4];    // lane quarter q: both halves read the other's value
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barriers must fit below the exchange area");

struct WideParams {
    DecodeParams p;
    int32_t row_tiles;
};

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, Bars *bars, int32_t *status) {
    return mbar_wait_bounded(bar, parity, &bars->abort_flag, status, FLAG_TIMEOUT, kTimeoutNs);
}
__device__ __forceinline__ bool aborted(Bars *bars) { return *(volatile int32_t *)&bars->abort_flag != 0; }

// Physical block of logical block `lb` of sequence b, or -1.
__device__ __forceinline__ int block_of(const DecodeParams &p, int b, int lb) {
    if (lb >= p.max_blocks) return -1;
    const int blk = p.block_table[(size_t)b * p.max_blocks + lb];
    return (blk >= 0 && blk < p.s.num_blocks) ? blk : -1;
}

__host__ __device__ constexpr int steps_of(int t0, int t1) { return (t1 - t0 + kStep - 1) / kStep; }

__global__ void __launch_bounds__(kThreads, 1)
decode_wide_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap o_map, const WideParams wp) {
    const DecodeParams &p = wp.p;
    const int half = blockIdx.x;             // 0/1: which 256 latent output dims
    const int g = blockIdx.y;                // query row tile
    const int stream = blockIdx.z;           // work stream (persistent over its items)
    const int rows_seq = p.q_len * p.s.H;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars *bars = (Bars *)(smem + kOffBar);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) WTRACE(11, 0);
#ifdef MLA_TRACE
    const unsigned cta_id = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    if (tid == 0 && cta_id < 2048) g_wcta[cta_id][0] = globaltimer();
#endif

    if (tid == 0) {
        mbar_init(&bars->full_a, 1);
        mbar_init(&bars->full_v, 1);
        mbar_init(&bars->empty_a, 1);
        mbar_init(&bars->empty_v, 1);
        mbar_init(&bars->tail_done, 1);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->p_full, kSoftmaxThreads);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->q_stage, 1);
        mbar_init(&bars->q_smem, 1);
        mbar_init(&bars->q_tmem, kSoftmaxThreads);
        mbar_init(&bars->qreg_free, kSoftmaxThreads);
        mbar_init(&bars->mma_fin, 1);
        for (int q = 0; q < 4; ++q) {
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
    // Each CTA asks L2 for its share of the query (a call input; only a cache hint),
    // so that the first work item's query load does not wait on DRAM.
    if (tid == 0) {
        const size_t q_bytes = (size_t)p.B * rows_seq * kD * 2;
        const size_t n_ctas = (size_t)gridDim.x * gridDim.y * gridDim.z;
        const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        const size_t share = ((q_bytes + n_ctas - 1) / n_ctas + 15) & ~(size_t)15;
        const size_t lo = cta * share;
        if (lo < q_bytes) {
            const size_t hi = min(q_bytes, lo + share);
            prefetch_l2((const uint8_t *)p.q + lo, (uint32_t)((hi - lo) & ~(size_t)15));
        }
    }
    // the set-up above overlaps the planner; its schedule is read only from here on.
    // The combine may launch from here: the planner has completed, so the combine can
    // read the schedule's split ranges before its own wait.
    pdl_wait();
    pdl_trigger();
#ifdef MLA_TRACE
    if (tid == 0 && cta_id < 2048) g_wcta[cta_id][1] = globaltimer();
#endif
    const int i0 = p.stream_start[stream], i1 = p.stream_start[stream + 1];
    if (i0 >= i1) {                          // no work for this stream (CTA-uniform)
        if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
        return;
    }

    if (warp == 0) {
        // ================================================= producer (+ L2 prefetch)
        // The warp runs converged; lane 0 waits and arms the barriers, one lane per box.
        const bool prefetcher = kPrefetchAhead > 0 && half == 0 && g == 0;
        int pi = i0, pt = 0, ahead = 0;
        auto advance_prefetch = [&]() {
            while (pi < i1 && ahead < kPrefetchAhead) {
                const WorkItem it = p.work[pi];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                if (pt >= nt) { ++pi; pt = 0; continue; }
                const int blk = block_of(p, it.b, it.t0 / kTile + pt);
                if (blk >= 0)       // the block's rows (index keys included: one contiguous range)
                    prefetch_l2((const __nv_bfloat16 *)p.latent + (size_t)blk * kTile * p.s.E(),
                                (uint32_t)kTile * p.s.E() * 2);
                ++pt;
                ++ahead;
            }
        };
        const int oob_row = p.s.num_blocks * kTile;   // past the end: TMA fills zeros
        int K = 0;
        bool ok = true;
        uint32_t tail_issued = 0;                      // partial-tile zeroings signalled
        for (int i = i0; i < i1 && ok; ++i) {
            const WorkItem it = p.work[i];
            const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
            const int L = p.seq_lens[it.b];
            const int ns = steps_of(it.t0, it.t1);
            for (int j = 0; j < ns; ++j, ++K) {
                // the step's two tiles: physical rows of each (a missing or bad block reads
                // zeros past the end; the softmax marks a bad block's rows NaN)
                int row0[2];
                int valid[2];
                for (int u = 0; u < 2; ++u) {
                    const int t = 2 * j + u;
                    valid[u] = t < nt ? min(kTile, L - (it.t0 + t * kTile)) : 0;
                    int blk = t < nt ? block_of(p, it.b, it.t0 / kTile + t) : -1;
                    if (t < nt && blk < 0 && lane == 0) raise_flag(p.status, FLAG_BAD_BLOCK);
                    row0[u] = blk >= 0 ? blk * kTile : oob_row;
                }
                // score-only blocks: free once the previous step's score MMAs over them completed
                if (K > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->empty_a, (K - 1) & 1, bars, p.status))) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_expect_tx(&bars->full_a, 10 * kBox);
                __syncwarp();
                if (lane < 10) {
                    const int u = lane / 5, c = score_only_block(half, lane % 5);
                    tma_load_2d(smem + kOffBuf + c * kCol + u * kBox, &kv_map, 64 * c, row0[u], &bars->full_a);
                }
                if (lane == 0) WTRACE(0, K);
                // own blocks: free once the previous step's PV completed
                if (K > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->empty_v, (K - 1) & 1, bars, p.status))) {
                    ok = false;
                    mbar_drain(&bars->full_a, K & 1);      // this step's score-only boxes are in flight
                    break;
                }
                if (lane == 0) mbar_expect_tx(&bars->full_v, 8 * kBox);
                __syncwarp();
                if (lane < 8) {
                    const int u = lane / 4, c = 4 * half + (lane % 4);
                    tma_load_2d(smem + kOffBuf + c * kCol + u * kBox, &kv_map, 64 * c, row0[u], &bars->full_v);
                }
                if (lane == 0) WTRACE(1, K);
                // a sequence's final partial block: once its own rows have landed, zero those
                // past the end so that P = 0 never meets stale (possibly non-finite) cache
                // bytes in PV (the scores of those slots are masked)
                const bool partial = (valid[0] > 0 && valid[0] < kTile) || (valid[1] > 0 && valid[1] < kTile);
                if (partial) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->full_v, K & 1, bars, p.status))) {
                        ok = false;
                        mbar_drain(&bars->full_a, K & 1);
                        break;
                    }
                    for (int u = 0; u < 2; ++u) {
                        if (valid[u] <= 0 || valid[u] >= kTile) continue;
                        const int jobs = (kTile - valid[u]) * 4 * 8;
                        for (int jb = lane; jb < jobs; jb += 32) {
                            const int rr = kTile * u + valid[u] + jb / 32, rem = jb % 32;
                            *(uint4 *)(smem + kOffBuf + (4 * half + (rem >> 3)) * kCol + sw128(rr, rem & 7)) =
                                make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->tail_done);
                    ++tail_issued;
                }
                if (lane == 0) {
                    if (prefetcher) ahead = max(0, ahead - 2);
                    if (prefetcher) advance_prefetch();
                }
            }
        }
        // drain: never leave a copy in flight into this CTA's shared memory
        if (K > 0) {
            mbar_drain(&bars->full_a, (K - 1) & 1);
            mbar_drain(&bars->full_v, (K - 1) & 1);
        }
        (void)tail_issued;
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer: lane 0 alone
        if (lane == 0) {
            constexpr uint32_t kIdQk = idesc_bf16(128, 128, false);
            constexpr uint32_t kIdPv = idesc_bf16(128, 256, true);
            const uint32_t qt = tmem + kColQ, d_s = tmem + kColS, d_o = tmem + kColO;
            const uint64_t qd = sdesc(smem_u32(smem + kOffQ), 16, 1024);
            const uint64_t bd = sdesc(smem_u32(smem + kOffBuf), 16, 1024);
            // MN-major V: 64-dim atoms 16 KB apart (column blocks), 8-token groups 1 KB apart
            const uint64_t vd = sdesc(smem_u32(smem + kOffBuf + 4 * half * kCol), kCol, 1024);
            bool ok = true;
            int K = 0;
            uint32_t tail_par = 0;
            int item_no = 0;
            for (int i = i0; i < i1 && ok; ++i, ++item_no) {
                const WorkItem it = p.work[i];
                const int L = p.seq_lens[it.b];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                const int ns = steps_of(it.t0, it.t1);
                if (!mbar_wait(&bars->q_tmem, item_no & 1, bars, p.status)) { ok = false; break; }
                for (int j = 0; j < ns; ++j, ++K) {
                    if (!mbar_wait(&bars->full_a, K & 1, bars, p.status)) { ok = false; break; }
                    WTRACE(2, K);
                    // S / P's tensor memory is free once the previous step's PV completed
                    if (K > 0 && !mbar_wait(&bars->pv_done, (K - 1) & 1, bars, p.status)) { ok = false; break; }
                    // the item's first step: Q's shared-memory part may still be landing
                    if (j == 0 && !mbar_wait(&bars->q_smem, item_no & 1, bars, p.status)) { ok = false; break; }
                    tc_fence_after();
                    // part 1: score-only blocks, Q from shared memory. K-step (k, s): Q slot k /
                    // column block score_only_block(k), 32-byte step s inside the swizzle atom
                    // (descriptor start addresses advance in 16-byte units)
#pragma unroll
                    for (int k = 0; k < kQSmemBlocks; ++k) {
                        const uint32_t cb = (uint32_t)score_only_block(half, k) * kCol;
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint64_t a = qd + (uint64_t)((k * kQBlock + 32 * s) >> 4);
                            const uint64_t b = bd + (uint64_t)((cb + 32 * s) >> 4);
                            if (k == 0 && s == 0) mma_ss_k<kIdQk, 0>(d_s, a, b);
                            else mma_ss_k<kIdQk, 1>(d_s, a, b);
                        }
                    }
                    mma_commit(&bars->empty_a);
                    WTRACE(3, K);
                    if (!mbar_wait(&bars->full_v, K & 1, bars, p.status)) { ok = false; break; }
                    WTRACE(4, K);
                    tc_fence_after();
                    // part 2: own blocks, Q from tensor memory (8 columns per K-step)
#pragma unroll
                    for (int k = 0; k < kQTmemBlocks; ++k) {
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            mma_ts_k<kIdQk, 1>(d_s, qt + 32 * k + 8 * s,
                                               bd + (uint64_t)(((4 * half + k) * kCol + 32 * s) >> 4));
                    }
                    mma_commit(&bars->s_full);
                    WTRACE(5, K);
                    // PV once the softmax stored P (and, for a partial tile, the producer
                    // zeroed its own rows past the end)
                    if (!mbar_wait(&bars->p_full, K & 1, bars, p.status)) { ok = false; break; }
                    WTRACE(6, K);
                    const int v0 = min(kTile, L - (it.t0 + 2 * j * kTile));
                    const int v1 = 2 * j + 1 < nt ? min(kTile, L - (it.t0 + (2 * j + 1) * kTile)) : 0;
                    if ((v0 > 0 && v0 < kTile) || (v1 > 0 && v1 < kTile)) {
                        if (!mbar_wait(&bars->tail_done, tail_par & 1u, bars, p.status)) { ok = false; break; }
                        tail_par ^= 1u;
                    }
                    tc_fence_after();
                    // K-step kk: P columns 8 kk (two bf16 tokens per column), V rows 16 kk
                    // (two 8-token groups, 2 KB)
#pragma unroll
                    for (int kk = 0; kk < kStep / 16; ++kk) {
                        if (kk == 0 && j == 0) mma_ts_k<kIdPv, 0>(d_o, d_s, vd);
                        else mma_ts_k<kIdPv, 1>(d_o, d_s + 8 * kk, vd + (uint64_t)(128 * kk));
                    }
                    mma_commit(&bars->pv_done);
                    mma_commit(&bars->empty_v);
                    WTRACE(7, K);
                }
            }
            mma_commit(&bars->mma_fin);
            mbar_wait(&bars->mma_fin, 0, bars, p.status);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ================================================= Q loads, softmax, epilogue
        // Warp w owns rows 32*(w%4)..+31 (its TMEM lane quarter) and half hs = (w-4)/4 of
        // the step: score columns 64*hs..+63 (tile hs), P columns 32*hs..+31, output
        // columns 128*hs..+127. Every branch around tcgen05.ld / tcgen05.st is warp-uniform.
        //
        // The Q region serves three uses in turn: staging the tensor-memory part of an
        // item's Q (TMA in, tcgen05.st out), the epilogue's output boxes, and Q's
        // shared-memory part that the score MMAs read. qreg_free completes once every
        // softmax thread is done with a staging or epilogue use; the TMA issuer (warp 4
        // lane 0) waits for it before loading into the region.
        const int wq = warp & 3;
        const int hs = (warp - 4) >> 2;
        const int row = 32 * wq + lane;
        const int row_seq = g * kRows + row;
        const bool row_valid = row_seq < rows_seq;
        const bool issuer = warp == 4 && lane == 0;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16);
        float *xchg = (float *)(smem + kOffXchg);
        bool ok = true;
        int K = 0, nx = 0, uses = 0, nstage = 0;
        // Swap one value per row with the other half of the row (bounded waits). The
        // tensor-memory fences order each side's tcgen05 accesses before the swap against
        // the other side's after it.
        auto exchange = [&](float v, float &other) -> bool {
            if (nx > 0 && !mbar_wait(&bars->xchg_read[wq], (nx - 1) & 1, bars, p.status)) return false;
            xchg[hs * 128 + row] = v;
            tc_fence_before();
            mbar_arrive(&bars->xchg_full[wq]);
            if (!mbar_wait(&bars->xchg_full[wq], nx & 1, bars, p.status)) return false;
            tc_fence_after();
            other = xchg[(hs ^ 1) * 128 + row];
            mbar_arrive(&bars->xchg_read[wq]);
            ++nx;
            return true;
        };
        // TMA of Q part `round` of work item `item` into the Q region (issuer only): round
        // 0 stages the tensor-memory part (the own latent blocks), round 1 loads the
        // shared-memory part (the score-only dims, in score_only_block order).
        auto issue_q = [&](int item, int round) -> bool {
            if (!issuer) return true;
            if (uses > 0 && !mbar_wait(&bars->qreg_free, (uses - 1) & 1, bars, p.status)) return false;
            const int qrow = p.work[item].b * rows_seq + g * kRows;
            if (round == 0) {
                mbar_expect_tx(&bars->q_stage, kQTmemBlocks * kQBlock);
                for (int k = 0; k < kQTmemBlocks; ++k)
                    tma_load_2d(smem + kOffQ + k * kQBlock, &q_map, 64 * (4 * half + k), qrow, &bars->q_stage);
            } else {
                mbar_expect_tx(&bars->q_smem, kQSmemBlocks * kQBlock);
                for (int k = 0; k < kQSmemBlocks; ++k)
                    tma_load_2d(smem + kOffQ + k * kQBlock, &q_map, 64 * score_only_block(half, k), qrow, &bars->q_smem);
            }
            return true;
        };
        // Staged Q -> tensor memory: thread (row, hs) moves blocks hs and hs + 2.
        auto load_q_tmem = [&](int item) -> bool {
            (void)item;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_stage, nstage & 1, bars, p.status))) return false;
            ++nstage;
#pragma unroll 1
            for (int k = hs; k < kQTmemBlocks; k += 2) {
                uint32_t v[32];
                const uint8_t *blk = smem + kOffQ + k * kQBlock;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 u = *(const uint4 *)(blk + sw128(row, ch));
                    v[4 * ch + 0] = u.x;
                    v[4 * ch + 1] = u.y;
                    v[4 * ch + 2] = u.z;
                    v[4 * ch + 3] = u.w;
                }
                TMEM_ST32(lane_addr + kColQ + 32 * k, v);
            }
            mbar_arrive(&bars->qreg_free);
            ++uses;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->q_tmem);
            return true;
        };
        ok = __all_sync(0xffffffffu, issue_q(i0, 0));
        ok = ok && load_q_tmem(i0);
        ok = ok && __all_sync(0xffffffffu, issue_q(i0, 1));
        for (int i = i0; i < i1 && ok; ++i) {
            const WorkItem it = p.work[i];
            const int L = p.seq_lens[it.b];
            const int t0 = it.t0, t1 = it.t1;
            const int nt = (t1 - t0 + kTile - 1) / kTile;
            const int ns = steps_of(t0, t1);
            const int last_vis = L - p.q_len + (row_valid ? row_seq / p.s.H : 0);
            float m_used = -CUDART_INF_F, l = 0.f;       // l: this half's share of the row sum
            bool bad_item = false;
            for (int t = 0; t < nt; ++t) bad_item |= block_of(p, it.b, t0 / kTile + t) < 0;
            for (int j = 0; j < ns && ok; ++j, ++K) {
                if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, K & 1, bars, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tid == 128) WTRACE(8, K);
                uint32_t sv[64];
                TMEM_LD32(lane_addr + kColS + 64 * hs, sv);
                TMEM_LD32(lane_addr + kColS + 64 * hs + 32, (sv + 32));
                tmem_wait_ld();
                const int tile_start = t0 + j * kStep + kTile * hs;
                const int n_vis = row_valid ? max(0, min(t1, last_vis + 1) - tile_start) : 0;
                // Scores stay unscaled where the scale is positive: the row max then commutes
                // with the scaling and each exponent argument is one fma. Hidden slots -> -inf.
                const bool pos_scale = p.scale_log2 > 0.f;
                const float cs = pos_scale ? p.scale_log2 : 1.f;
                if (!pos_scale || __any_sync(0xffffffffu, n_vis < kTile)) {
#pragma unroll
                    for (int jj = 0; jj < 64; ++jj) {
                        const float v = pos_scale ? __uint_as_float(sv[jj]) : __uint_as_float(sv[jj]) * p.scale_log2;
                        sv[jj] = __float_as_uint(jj < n_vis ? v : -CUDART_INF_F);
                    }
                }
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int jj = 0; jj < 64; ++jj) mx = fmaxf(mx, __uint_as_float(sv[jj]));
                mx *= cs;
                // the row's max over both halves; after it, both halves have read their S
                // columns, so P may be stored over them
                {
                    float other = -CUDART_INF_F;
                    if (!__all_sync(0xffffffffu, exchange(mx, other))) { ok = false; break; }
                    mx = fmaxf(mx, other);
                }
                if (tid == 128) WTRACE(9, K);
                float alpha = 1.f;
                bool rescale = false;
                const float m_new = fmaxf(m_used, mx);
                if (m_new > m_used + 8.f) {
                    alpha = exp2f(m_used - m_new);        // 0 when nothing was accumulated yet
                    m_used = m_new;
                    rescale = j > 0;
                }
                const float nmb = m_used == -CUDART_INF_F ? -CUDART_INF_F : -m_used;
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const float a = ex2(fmaf(__uint_as_float(sv[2 * jj]), cs, nmb));
                    const float c = ex2(fmaf(__uint_as_float(sv[2 * jj + 1]), cs, nmb));
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(a, c);
                    pk[jj] = *(const uint32_t *)&hh;
                    sum0 += a;             // fp32 row sum: the LSE does not see the rounding of P
                    sum1 += c;
                }
                l = l * alpha + (sum0 + sum1);
                // O *= alpha: the previous step's PV completed before these scores were
                // computed (the MMA thread issues a step's score MMAs after it)
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 4 * hs; c < 4 * hs + 4; ++c) {
                        uint32_t ov[32];
                        TMEM_LD32(lane_addr + kColO + 32 * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
                        TMEM_ST32(lane_addr + kColO + 32 * c, ov);
                    }
                }
                TMEM_ST32(lane_addr + kColS + 32 * hs, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->p_full);
                if (tid == 128) WTRACE(10, K);
            }
            // ---- end of this item. The Q region is free (the item's last score MMAs have
            // completed): stage the next item's tensor-memory Q while the last PV runs, then
            // write this item's output through the region, then load the next item's
            // shared-memory Q part.
            const bool have_next = i + 1 < i1;
            if (ok && have_next) ok = __all_sync(0xffffffffu, issue_q(i + 1, 0));
            if (ok && ns > 0) ok = __all_sync(0xffffffffu, mbar_wait(&bars->pv_done, (K - 1) & 1, bars, p.status));
            float l_other = 0.f;
            if (ok) ok = __all_sync(0xffffffffu, exchange(l, l_other));
            const float l_row = l + l_other;
            tc_fence_after();
            if (ok && have_next) ok = load_q_tmem(i + 1);
            if (ok && have_next)
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->qreg_free, (uses - 1) & 1, bars, p.status));
            const bool bad = aborted(bars) || !ok || bad_item;
            // Epilogue: O / l -> partial slot i, rounded to bf16; [32 rows x 64 dims] boxes
            // (128B-swizzled) through the region, one TMA store each; rows past the
            // sequence's rows are clipped by the tensor map.
            if (ok) {
                const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                const uint64_t keep = l2_policy_evict_last();
                uint8_t *boxes = smem + kOffQ + (warp - 4) * kEpiBoxes * kEpiBoxBytes;
                const int y = g * kRows + 32 * wq;
                const bool store = y < rows_seq;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    const int bi = c % kEpiBoxes;
                    if (bi == 0 && c > 0) {
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
                    }
                    uint8_t *box = boxes + bi * kEpiBoxBytes;
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t ov[32];
                        TMEM_LD32(lane_addr + kColO + 128 * hs + 64 * c + 32 * hh, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t pk4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                                    __uint_as_float(ov[8 * q + 2 * e]) * inv, __uint_as_float(ov[8 * q + 2 * e + 1]) * inv);
                                pk4[e] = *(const uint32_t *)&h2;
                            }
                            *(uint4 *)(box + sw128(lane, 4 * hh + q)) = make_uint4(pk4[0], pk4[1], pk4[2], pk4[3]);
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
            if (ok && have_next) ok = __all_sync(0xffffffffu, issue_q(i + 1, 1));
        }
        if (lane == 0) bulk_wait_all();   // this warp's output stores have landed
    }
    tc_fence_before();
    __syncthreads();
#ifdef MLA_TRACE
    if (tid == 0 && cta_id < 2048) g_wcta[cta_id][2] = globaltimer();
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

// 2-D bf16 map over the first 576 columns of a row-major [rows, row_elems] matrix,
// 128-byte swizzled boxes of [box_rows, 64]. Rows past the end read as zero.
static bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows, uint64_t row_elems) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D bf16 map over the partial outputs [slots, rows_seq, r], boxes of [32 rows x 64
// dims] with the 128-byte swizzle (stores clip rows >= rows_seq).
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

}  // namespace wide

cudaError_t launch_decode_wide(const DecodeParams &p, int32_t max_work, cudaStream_t st) {
    wide::WideParams wp;
    wp.p = p;
    wp.row_tiles = (p.q_len * p.s.H + wide::kRows - 1) / wide::kRows;
    CUtensorMap kv_map, q_map, o_map;
    if (!wide::make_map(&kv_map, p.latent, (uint64_t)p.s.num_blocks * p.s.bs, wide::kTile, (uint64_t)p.s.E()))
        return cudaErrorInvalidValue;
    const int rows_seq = p.q_len * p.s.H;
    if (!wide::make_map(&q_map, p.q, (uint64_t)p.B * rows_seq, wide::kRows, wide::kD)) return cudaErrorInvalidValue;
    if (!wide::make_out_map(&o_map, p.part_o, p.s.r, rows_seq, max_work)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(wide::decode_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)wide::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(2, wp.row_tiles, p.streams);
    return launch_pdl(wide::decode_wide_kernel, grid, dim3(wide::kThreads), wide::kSmemBytes, st, kv_map, q_map, o_map,
                      wp);
}

}  // namespace mla

#ifdef MLA_TRACE
extern "C" int mla_wide_trace_read(long long *events) {
    return (int)cudaMemcpyFromSymbol(events, mla::wide::g_wtrace, sizeof(mla::wide::g_wtrace));
}
extern "C" int mla_wide_cta_read(unsigned long long *times) {
    return (int)cudaMemcpyFromSymbol(times, mla::wide::g_wcta, sizeof(mla::wide::g_wcta));
}
#endif
