// Tensor-core (tcgen05 / TMEM / TMA) split-KV decode for the bf16 latent cache of
// the DeepSeek-V3 shape (kv_lora_rank 512, rope 64, block size 64), run by pairs of
// CTAs (2-CTA clusters) that take turns computing the scores.
//
// Why a pair. The latent output of 128 query rows x 512 dims is 256 KB of fp32, the
// whole tensor memory of one SM, so the output is split across two CTAs: CTA h owns
// latent dims [256h, 256h + 256). Every 64-token tile needs the scores S of all 128
// rows over all 576 dims, but computing them in both CTAs doubles the most expensive
// MMA work (36 M128 N64 K16 MMAs a tile, whose cost per instruction hardly depends on
// N), and reading every tile in both CTAs doubles the L2 -> SM traffic. Here the tiles
// of a stream alternate: tile T is "owned" by CTA T % 2, which alone loads all of the
// tile and computes S, the softmax and P; the other CTA loads only its 256 V dims of
// the tile and receives P (bf16 [128 x 64], 16 KB) in its own shared memory, written
// by the softmax threads with 16-byte st.async stores that complete transaction bytes
// on the receiver's barrier. Both then accumulate O += P . V for their own dims.
//
// The softmax base. Both CTAs accumulate into outputs that must share one running
// maximum per row. The owner of tile T derives it from the base after tile T-1 (held
// by the other CTA, which owned T-1) and the row maxima of tile T; it sends the new
// base (512 bytes) to the other CTA right after computing it, so the bases form a
// chain that alternates between the two CTAs, one hop per tile, off the MMA path.
// The base is raised lazily (only when the row max grows by more than 8, so P <= 256),
// and both CTAs rescale their own outputs by the same factors. Row sums are kept per
// CTA (each over the tiles it owns, rescaled at every tile) and added at the end of a
// work item through a second small message.
//
// Per CTA, per tile T it owns:
//   TMA     its 4 V boxes [64 tokens x 64 dims] + the 5 score-only boxes (the other
//           CTA's latent dims and the rope key), 128B-swizzled
//   MMA     S[128 x 64] = Q[128 x 576] . K[64 x 576]^T  (24 K-steps with Q in tensor
//           memory, 12 with Q in shared memory)
//   softmax S -> registers, causal/length mask, row max (two warps per row), base,
//           P = 2^(s*scale*log2e - base) rounded to bf16 into the CTA's P buffer
//           and (st.async) into the other CTA's
//   MMA     O[128 x 256] += P[128 x 64] . V[64 x 256]  (8 M128 N128 K16 MMAs)
// and per tile it does not own: TMA of its 4 V boxes, the base message (rescale),
// then the same PV from the received P.
//
// Roles: warp 0 = V producer (+ L2 prefetch, + zeroing of a partial tile's slots past
// the end), warp 10 = score-only producer; warp 1 = TMEM owner, lane 0 issues the
// score MMAs; warp 11, lane 0, the PV MMAs; warps 2..9 = Q loads,
// softmax, messages and the epilogue (warp w reads TMEM lanes 32*(w%4)..+31, half
// (w-2)/4 of each row). Every wait is bounded (2 s); a wait that gives up records
// FLAG_TIMEOUT and the CTA winds down without trapping. Both CTAs wait for every
// message and copy addressed to them before the final cluster barrier, so no
// shared-memory write of one CTA can land after the other has exited.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>
#include <string.h>

namespace mla {
namespace pair {

using namespace ptx;

constexpr int kThreads = 384;          // warp 0 V producer, 1 score MMAs, 2..9 softmax, 10 score-only
                                       // producer, 11 PV MMAs
constexpr int kPvWarp = 11;
constexpr int kTWarp = 10;
constexpr int kSoftmaxThreads = 256;
constexpr int kTile = 64;              // tokens per tile == cache block size
constexpr int kRows = 128;             // query rows per CTA (MMA M)
constexpr int kD = 576;                // r + d_R
constexpr int kNV = 3;                 // V segments in flight (every tile)
constexpr int kNT = 1;                 // score-only segments in flight (owned tiles)
constexpr uint32_t kBox = kTile * 128;                 // [64 tokens x 64 dims] bf16: 8 KB
constexpr uint32_t kVSeg = 4 * kBox;                   // the CTA's 256 V dims: 32 KB
constexpr uint32_t kTSeg = 5 * kBox;                   // other half's dims + rope: 40 KB
constexpr uint32_t kQBlock = kRows * 128;              // [128 rows x 64 dims] bf16: 16 KB
constexpr int kQTmemBlocks = 6, kQSmemBlocks = 3;      // Q dims 0..383 in TMEM, 384..575 in smem
constexpr int kQRounds = (kQTmemBlocks + kQSmemBlocks - 1) / kQSmemBlocks;
constexpr uint32_t kPBytes = kRows * 128;              // P [128 rows x 64 tokens] bf16: 16 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffP = kOffQ + kQSmemBlocks * kQBlock;     // 48 KB
constexpr uint32_t kOffV = kOffP + 2 * kPBytes;                // 80 KB
constexpr uint32_t kOffT = kOffV + kNV * kVSeg;                // 176 KB
constexpr uint32_t kOffBar = kOffT + kNT * kTSeg;              // 216 KB
constexpr uint32_t kOffXchg = kOffBar + 512;                   // [2][128] fp32: row halves
constexpr uint32_t kOffBmsg = kOffXchg + 1024;                 // [128] fp32: received bases
constexpr uint32_t kOffLmsg = kOffBmsg + 512;                  // [2][128] fp32: received row sums
constexpr uint32_t kSmemBytes = kOffLmsg + 1024 + 1024;        // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffV % 1024 == 0 && kOffT % 1024 == 0 && kOffP % 1024 == 0, "1 KB alignment of MMA operands");
constexpr uint32_t kColO = 0, kColS = 256, kColQ = 320;       // tensor-memory columns (512 allocated)
constexpr uint32_t kEpiBoxBytes = 32 * 128;                    // epilogue box: [32 rows x 64 dims] bf16
constexpr int kQkSplit = 24;                                   // K-steps [0,24): A from TMEM; [24,36): smem
constexpr unsigned long long kTimeoutNs = 2000000000ull;       // 2 s bounded-wait safety net
#ifndef MLA_PAIR_PREFETCH_AHEAD
#define MLA_PAIR_PREFETCH_AHEAD 4
#endif
constexpr int kPrefetchAhead = MLA_PAIR_PREFETCH_AHEAD;        // blocks prefetched into L2 ahead

// Pipeline timestamps for performance analysis, compiled only with -DMLA_TRACE:
// clock64 at each hand-off of both CTAs of one pair (stream MLA_TRACE_STREAM, row
// tile 0) for its first kTraceTiles tiles, plus each CTA's (clock64, globaltimer) at
// entry to align the two clocks. Product builds contain none of it.
#ifdef MLA_TRACE
#ifndef MLA_TRACE_STREAM
#define MLA_TRACE_STREAM 0
#endif
constexpr int kTraceTiles = 64;
__device__ long long g_ptrace[2][16][kTraceTiles];
__device__ long long g_pstart[2][2];
#define PTRACE(ev, tile)                                                                                   \
    do {                                                                                                   \
        if (blockIdx.y == 0 && blockIdx.z == MLA_TRACE_STREAM && (tile) < kTraceTiles) g_ptrace[h][ev][tile] = clock64(); \
    } while (0)
#else
#define PTRACE(ev, tile) \
    do {                 \
    } while (0)
#endif
// events: 0 V boxes issued, 1 score-only boxes issued (producer), 2 QK first half
// issued, 3 QK second half issued, 4 PV issued (MMA), 5 S seen, 6 row max agreed,
// 7 P buffer free, 8 P copy issued (owned tile), 9 base received (other's tile),
// 10 ready arrived (softmax)

struct Bars {
    uint64_t v_full[kNV], v_empty[kNV], v_tail[kNV];
    uint64_t t_full[kNT], t_empty[kNT], t_tail[kNT];
    uint64_t s_full, s_free;
    uint64_t ready[2];        // softmax done with tile T (index T % 2): P written / O rescaled
    uint64_t p_rx;            // the other CTA's P of one of its tiles landed here
    uint64_t pv_done[2];      // PV of tile T (index T % 2) completed
    uint64_t rbuf_free;       // the other CTA's PV of one of this CTA's tiles completed
    uint64_t bmsg;            // the other CTA's base for one of its tiles landed
    uint64_t lmsg[2];         // the other CTA's row sums at the end of a work item (item % 2)
    uint64_t q_stage, q_smem, q_tmem, qreg_free;
    uint64_t mma_fin, pv_fin;
    uint64_t xchg_full, xchg_read;
    int32_t pv_issued;        // tiles whose PV MMAs have been issued (PV issuer -> score issuer)
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barriers must fit below the exchange area");

struct PairParams {
    DecodeParams p;
    int32_t row_tiles;
};

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, Bars *bars, int32_t *status) {
    return mbar_wait_bounded(bar, parity, &bars->abort_flag, status, FLAG_TIMEOUT, kTimeoutNs);
}
__device__ __forceinline__ bool aborted(Bars *bars) { return *(volatile int32_t *)&bars->abort_flag != 0; }

// Physical block of logical tile `lb` of sequence b, or -1.
__device__ __forceinline__ int block_of(const DecodeParams &p, int b, int lb) {
    if (lb >= p.max_blocks) return -1;
    const int blk = p.block_table[(size_t)b * p.max_blocks + lb];
    return (blk >= 0 && blk < p.s.num_blocks) ? blk : -1;
}

__global__ void __launch_bounds__(kThreads, 1)
decode_pair_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap o_map, const PairParams pp) {
    const DecodeParams &p = pp.p;
    const uint32_t h = cluster_ctarank();    // 0/1: which 256 latent output dims
    const uint32_t peer = h ^ 1u;
    const int g = blockIdx.y;                // query row tile
    const int stream = blockIdx.z;           // work stream (persistent over its items)
    pdl_trigger();
    const int rows_seq = p.q_len * p.s.H;
#ifdef MLA_TRACE
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == MLA_TRACE_STREAM) {
        g_pstart[h][0] = clock64();
        g_pstart[h][1] = (long long)globaltimer();
    }
#endif

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    Bars *bars = (Bars *)(smem + kOffBar);
    float *bbuf = (float *)(smem + kOffBmsg);
    float *lbuf = (float *)(smem + kOffLmsg);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kNV; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->v_tail[s], 1);
        }
        for (int s = 0; s < kNT; ++s) {
            mbar_init(&bars->t_full[s], 1);
            mbar_init(&bars->t_empty[s], 1);
            mbar_init(&bars->t_tail[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, kSoftmaxThreads);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->ready[i], kSoftmaxThreads);
            mbar_init(&bars->pv_done[i], 1);
            mbar_init(&bars->lmsg[i], 1);
        }
        mbar_init(&bars->p_rx, 1);
        mbar_init(&bars->rbuf_free, 1);
        mbar_init(&bars->bmsg, 1);
        mbar_init(&bars->q_stage, 1);
        mbar_init(&bars->q_smem, 1);
        mbar_init(&bars->q_tmem, kSoftmaxThreads);
        mbar_init(&bars->qreg_free, kSoftmaxThreads);
        mbar_init(&bars->mma_fin, 1);
        mbar_init(&bars->pv_fin, 1);
        bars->pv_issued = 0;
        mbar_init(&bars->xchg_full, kSoftmaxThreads);
        mbar_init(&bars->xchg_read, kSoftmaxThreads);
        bars->abort_flag = 0;
        // phase 0 of every barrier the other CTA completes by transaction bytes is armed
        // here; each later phase is armed by its consumer once the previous one completed
        mbar_expect_tx(&bars->p_rx, kPBytes);
        mbar_expect_tx(&bars->bmsg, kRows * 4);
        mbar_expect_tx(&bars->lmsg[0], kRows * 4);
        mbar_expect_tx(&bars->lmsg[1], kRows * 4);
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
    // the other CTA's barriers are initialised before any message is sent to it
    cluster_sync();
    const uint32_t tmem = bars->tmem_base;
    // the set-up above overlaps the planner; its schedule is read only from here on
    pdl_wait();
    const int i0 = p.stream_start[stream], i1 = p.stream_start[stream + 1];
    if (i0 >= i1) {                          // no work for this stream (same in both CTAs)
        if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
        return;
    }
    auto owned = [&](int T) { return (uint32_t)(T & 1) == h; };

    if (warp == 0 || warp == kTWarp) {
        // ================================================= producers (+ L2 prefetch)
        // Warp 0 loads the V boxes of every tile (lanes 0..3) and prefetches into L2;
        // warp 10 loads the score-only boxes of the owned tiles (lanes 0..4), so that
        // neither waits for the other's ring. Lane 0 waits and arms.
        const bool vrole = warp == 0;
        const bool prefetcher = vrole && kPrefetchAhead > 0 && h == 0 && g == 0;
        int pi = i0, pt = 0, ahead = 0;
        auto advance_prefetch = [&]() {
            while (pi < i1 && ahead < kPrefetchAhead) {
                const WorkItem it = p.work[pi];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                if (pt >= nt) { ++pi; pt = 0; continue; }
                const int blk = block_of(p, it.b, it.t0 / kTile + pt);
                if (blk >= 0)
                    prefetch_l2((const __nv_bfloat16 *)p.latent + (size_t)blk * kTile * p.s.E(),
                                (uint32_t)kTile * p.s.E() * 2);
                ++pt;
                ++ahead;
            }
        };
        int T = 0;
        bool ok = true;
        for (int i = i0; i < i1 && ok; ++i) {
            const WorkItem it = p.work[i];
            const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
            const int L = p.seq_lens[it.b];
            int next_blk = block_of(p, it.b, it.t0 / kTile);
            for (int t = 0; t < nt; ++t, ++T) {
                int blk = next_blk;
                if (t + 1 < nt) next_blk = block_of(p, it.b, it.t0 / kTile + t + 1);
                if (blk < 0) {            // the softmax marks the item's rows NaN
                    if (lane == 0 && vrole) raise_flag(p.status, FLAG_BAD_BLOCK);
                    blk = 0;
                }
                const bool own = owned(T);
                const int vs = T % kNV;
                uint8_t *vseg = smem + kOffV + vs * kVSeg;
                if (vrole) {
                    if (T >= kNV &&
                        !__all_sync(0xffffffffu, mbar_wait(&bars->v_empty[vs], ((T - kNV) / kNV) & 1, bars, p.status))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_expect_tx(&bars->v_full[vs], kVSeg);
                    __syncwarp();
                    if (lane < 4)
                        tma_load_2d(vseg + lane * kBox, &kv_map, 64 * (4 * (int)h + lane), blk * kTile, &bars->v_full[vs]);
                    if (lane == 0) PTRACE(0, T);
                }
                const int k = T >> 1, ts = k % kNT;
                uint8_t *tseg = smem + kOffT + ts * kTSeg;
                if (own && !vrole) {
                    if (k >= kNT &&
                        !__all_sync(0xffffffffu, mbar_wait(&bars->t_empty[ts], ((k - kNT) / kNT) & 1, bars, p.status))) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_expect_tx(&bars->t_full[ts], kTSeg);
                    __syncwarp();
                    if (lane < 5) {
                        const int d = lane < 4 ? 4 * (1 - (int)h) + lane : 8;
                        tma_load_2d(tseg + lane * kBox, &kv_map, 64 * d, blk * kTile, &bars->t_full[ts]);
                    }
                    if (lane == 0) PTRACE(1, T);
                }
                // a sequence's final partial block: once it has landed, zero the slots past
                // the end so that P = 0 never meets stale (possibly non-finite) cache bytes
                const int valid = min(kTile, L - (it.t0 + t * kTile));
                if (valid < kTile && vrole) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[vs], (T / kNV) & 1, bars, p.status))) {
                        ok = false;
                        ++T;                   // this tile's boxes are in flight: drained below
                        break;
                    }
                    for (int jb = lane; jb < (kTile - valid) * 4 * 8; jb += 32) {
                        const int rr = valid + jb / 32, rem = jb % 32;
                        *(uint4 *)(vseg + (rem >> 3) * kBox + sw128(rr, rem & 7)) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->v_tail[vs]);
                }
                if (valid < kTile && !vrole) {
                    if (own) {
                        if (!__all_sync(0xffffffffu, mbar_wait(&bars->t_full[ts], (k / kNT) & 1, bars, p.status))) {
                            ok = false;
                            ++T;                   // this tile's boxes are in flight: drained below
                            break;
                        }
                        for (int jb = lane; jb < (kTile - valid) * 5 * 8; jb += 32) {
                            const int rr = valid + jb / 40, rem = jb % 40;
                            *(uint4 *)(tseg + (rem >> 3) * kBox + sw128(rr, rem & 7)) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->t_tail[ts]);
                    }
                }
                if (lane == 0 && prefetcher) {   // L2 prefetch after this tile's own loads
                    if (ahead > 0) --ahead;
                    advance_prefetch();
                }
            }
        }
        // drain: never leave a copy in flight into this CTA's shared memory
        if (vrole) {
            for (int u = T - kNV; u < T; ++u)
                if (u >= 0) mbar_drain(&bars->v_full[u % kNV], (u / kNV) & 1);
        } else {
            for (int u = T - 2 * kNT; u < T; ++u)
                if (u >= 0 && owned(u)) mbar_drain(&bars->t_full[(u >> 1) % kNT], ((u >> 1) / kNT) & 1);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kPvWarp) {
        // ================================================= MMA issuers (lane 0 of each)
        // Warp 1 issues the score MMAs of this CTA's owned tiles, warp kPvWarp the PV of
        // every tile, each in tile order as soon as its inputs are there (one issuer
        // for both held the PV of a tile back behind the next tile's score MMAs). Every
        // barrier phase is observed in order, each right after the one before it
        // completed, so a parity test never sees a barrier two phases away: a V slot's
        // phases are observed alternately by the two issuers (the scores of an owned
        // tile, the PV of the other CTA's), and the scores of tile T wait until PV(T-3),
        // the slot's previous user, was issued (published in pv_issued). Each issuer
        // toggles its own parity bit of a slot's tail barrier for every partial tile that
        // passes through the slot, observed by it or not.
        if (lane == 0) {
            const bool is_pv = warp == kPvWarp;
            const uint32_t d_o = tmem + kColO, d_s = tmem + kColS, qt = tmem + kColQ;
            constexpr uint32_t kIdQk = idesc_bf16(128, 64, false);
            constexpr uint32_t kIdPv = idesc_bf16(128, 128, true);
            volatile int32_t *pv_issued = &bars->pv_issued;
            bool ok = true;
            uint32_t vt_par = 0, tt_par = 0;      // bit s: parity of the partial tiles passed in slot s
            int T = 0, own_items = 0;
            for (int i = i0; i < i1 && ok; ++i) {
                const WorkItem it = p.work[i];
                const int nt = (it.t1 - it.t0 + kTile - 1) / kTile;
                const int L = p.seq_lens[it.b];
                const bool has_own = nt >= 2 || owned(T);
                bool q_seen = false;              // this item's Q observed (score issuer)
                for (int t = 0; t < nt && ok; ++t, ++T) {
                    const bool own = owned(T);
                    const int vs = T % kNV;
                    const int valid = min(kTile, L - (it.t0 + t * kTile));
                    const bool partial = valid < kTile;
                    if (is_pv) {
                        // ---- PV of tile T
                        ok = mbar_wait(&bars->ready[T & 1], (T >> 1) & 1, bars, p.status);
                        if (ok && !own) {
                            ok = mbar_wait(&bars->p_rx, (T >> 1) & 1, bars, p.status) &&
                                 mbar_wait(&bars->v_full[vs], (T / kNV) & 1, bars, p.status);
                            if (ok && partial) ok = mbar_wait(&bars->v_tail[vs], (vt_par >> vs) & 1u, bars, p.status);
                        }
                        if (partial) vt_par ^= 1u << vs;
                        if (!ok) break;
                        if (!own) {
                            mbar_expect_tx(&bars->p_rx, kPBytes);   // arm the next copy's phase
                            // P arrived by the other CTA's generic-proxy remote stores; the MMAs
                            // read it through the async proxy
                            fence_proxy_async();
                        }
                        tc_fence_after();
                        const uint64_t a0 = sdesc(smem_u32(smem + kOffP + (T & 1) * kPBytes), 16, 1024);
                        const uint64_t b0 = sdesc(smem_u32(smem + kOffV + vs * kVSeg), kBox, 1024);
                        // K-step k: 16 tokens (A +32 B, B +2 KB); N halves 2 V boxes (16 KB) apart
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t a = a0 + (uint64_t)(2 * k), b = b0 + (uint64_t)(128 * k);
                            if (t == 0 && k == 0) {
                                mma_ss_k<kIdPv, 0>(d_o, a, b);
                                mma_ss_k<kIdPv, 0>(d_o + 128, a, b + 1024);
                            } else {
                                mma_ss_k<kIdPv, 1>(d_o, a, b);
                                mma_ss_k<kIdPv, 1>(d_o + 128, a, b + 1024);
                            }
                        }
                        mma_commit(&bars->pv_done[T & 1]);
                        mma_commit(&bars->v_empty[vs]);
                        if (!own) mma_commit_mc(&bars->rbuf_free, (uint16_t)(1u << peer));
                        *pv_issued = T + 1;
                        PTRACE(4, T);
                    } else {
                        // ---- QK of tile T, if this CTA owns it
                        const int k = T >> 1, ts = k % kNT;
                        if (!own) {
                            if (partial) vt_par ^= 1u << vs;
                            continue;
                        }
                        if (!q_seen) {
                            ok = mbar_wait(&bars->q_tmem, own_items & 1, bars, p.status) &&
                                 mbar_wait(&bars->q_smem, own_items & 1, bars, p.status);
                            q_seen = true;
                        }
                        // the V slot's previous user, PV(T - 3), was issued
                        if (ok && *pv_issued <= T - kNV) {
                            const unsigned long long tw0 = globaltimer();
                            for (uint32_t it2 = 0; *pv_issued <= T - kNV; ++it2) {
                                if ((it2 & 63u) == 63u && (aborted(bars) || globaltimer() - tw0 > kTimeoutNs)) {
                                    if (!aborted(bars)) {
                                        atomicExch(&bars->abort_flag, 1);
                                        raise_flag(p.status, FLAG_TIMEOUT);
                                    }
                                    ok = false;
                                    break;
                                }
                                __nanosleep(32);
                            }
                        }
                        ok = ok && mbar_wait(&bars->t_full[ts], (k / kNT) & 1, bars, p.status) &&
                             mbar_wait(&bars->v_full[vs], (T / kNV) & 1, bars, p.status) &&
                             (k == 0 || mbar_wait(&bars->s_free, (k - 1) & 1, bars, p.status));
                        if (ok && partial)
                            ok = mbar_wait(&bars->t_tail[ts], (tt_par >> ts) & 1u, bars, p.status) &&
                                 mbar_wait(&bars->v_tail[vs], (vt_par >> vs) & 1u, bars, p.status);
                        if (partial) {
                            tt_par ^= 1u << ts;
                            vt_par ^= 1u << vs;
                        }
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t vd = sdesc(smem_u32(smem + kOffV + vs * kVSeg), 16, 1024);
                        const uint64_t td = sdesc(smem_u32(smem + kOffT + ts * kTSeg), 16, 1024);
                        const uint64_t qd = sdesc(smem_u32(smem + kOffQ), 16, 1024);
                        // K box d of the tile: this CTA's V dims live in the V segment, the rest
                        // (the other half's latent dims, then the rope key) in the T segment
                        auto kdesc = [&](int j) -> uint64_t {
                            const int d = j >> 2;
                            const uint32_t off = 32u * (j & 3);
                            if ((uint32_t)(d >> 2) == h && d < 8) return vd + (uint64_t)(((d & 3) * kBox + off) >> 4);
                            const int ti = d < 8 ? (d & 3) : 4;
                            return td + (uint64_t)((ti * kBox + off) >> 4);
                        };
                        mma_ts_k<kIdQk, 0>(d_s, qt, kdesc(0));
#pragma unroll
                        for (int j = 1; j < kQkSplit; ++j) mma_ts_k<kIdQk, 1>(d_s, qt + 8 * j, kdesc(j));
                        PTRACE(2, T);
#pragma unroll
                        for (int j = kQkSplit; j < 36; ++j)
                            mma_ss_k<kIdQk, 1>(
                                d_s, qd + (uint64_t)((((j >> 2) - kQTmemBlocks) * kQBlock + 32 * (j & 3)) >> 4), kdesc(j));
                        mma_commit(&bars->s_full);
                        mma_commit(&bars->t_empty[ts]);
                        PTRACE(3, T);
                    }
                }
                if (has_own) ++own_items;
            }
            uint64_t *fin = is_pv ? &bars->pv_fin : &bars->mma_fin;
            mma_commit(fin);
            mbar_wait(fin, 0, bars, p.status);
        }
        __syncwarp();
    } else {
        // ================================================= Q loads, softmax, messages, epilogue
        // Warps 2..9: warp w owns rows 32*(w%4)..+31 (its TMEM lane quarter) and half
        // hs = (w-2)/4 of each row: score columns 32*hs..+31, output columns 128*hs..+127.
        // Every branch around tcgen05.ld / tcgen05.st is warp-uniform.
        const int wq = warp & 3;
        const int hs = (warp - 2) >> 2;
        const int row = 32 * wq + lane;
        const int row_seq = g * kRows + row;
        const bool row_valid = row_seq < rows_seq;
        const bool issuer = warp == 2 && lane == 0;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16);
        float *xchg = (float *)(smem + kOffXchg);
        const uint32_t peer_bbuf = mapa(smem_u32(bbuf + row), peer);
        const uint32_t peer_bmsg = mapa(smem_u32(&bars->bmsg), peer);
        const uint32_t peer_pbase = mapa(smem_u32(smem + kOffP), peer);
        const uint32_t peer_prx = mapa(smem_u32(&bars->p_rx), peer);
        bool ok = true;
        int T = 0, nx = 0, uses = 0, nstage = 0;
        int n_own_sent = 0;                  // P copies sent to the other CTA
        auto exchange = [&](float v, float &other) -> bool {
            if (nx > 0 && !mbar_wait(&bars->xchg_read, (nx - 1) & 1, bars, p.status)) return false;
            xchg[hs * 128 + row] = v;
            mbar_arrive(&bars->xchg_full);
            if (!mbar_wait(&bars->xchg_full, nx & 1, bars, p.status)) return false;
            other = xchg[(hs ^ 1) * 128 + row];
            mbar_arrive(&bars->xchg_read);
            ++nx;
            return true;
        };
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
            mbar_expect_tx(bar, (uint32_t)n * kQBlock);
            for (int k = 0; k < n; ++k) tma_load_2d(smem + kOffQ + k * kQBlock, &q_map, 64 * (first + k), qrow, bar);
            return true;
        };
        auto stage_q = [&](int round) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->q_stage, nstage & 1, bars, p.status))) return false;
            ++nstage;
            const int first = round * kQSmemBlocks;
            const int n = min(kQSmemBlocks, kQTmemBlocks - first);
#pragma unroll 1
            for (int k = hs; k < n; k += 2) {
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
                TMEM_ST32(lane_addr + kColQ + 32 * (first + k), v);
            }
            mbar_arrive(&bars->qreg_free);
            ++uses;
            return true;
        };
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
        // O *= alpha (per row) on this thread's 128 output columns, once PV(T-1) landed
        auto rescale_o = [&](int Tprev, float alpha) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[Tprev & 1], (Tprev >> 1) & 1, bars, p.status))) return false;
            tc_fence_after();
#pragma unroll 1
            for (int c = 4 * hs; c < 4 * hs + 4; ++c) {
                uint32_t ov[32];
                TMEM_LD32(lane_addr + kColO + 32 * c, ov);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 32; ++q) ov[q] = __float_as_uint(__uint_as_float(ov[q]) * alpha);
                TMEM_ST32(lane_addr + kColO + 32 * c, ov);
            }
            tmem_wait_st();
            return true;
        };
        // Q is loaded only for the items of which this CTA owns a tile (their QK
        // observes one Q phase per such item, in order)
        auto has_own_tile = [&](int item, int T_first) {
            const WorkItem w = p.work[item];
            return (w.t1 - w.t0 + kTile - 1) / kTile >= 2 || owned(T_first);
        };
        if (has_own_tile(i0, 0)) {
            ok = __all_sync(0xffffffffu, issue_q(i0, 0));
            ok = ok && load_q_tmem(i0);
            ok = ok && __all_sync(0xffffffffu, issue_q(i0, kQRounds));
        }
        int item_no = 0;
        for (int i = i0; i < i1 && ok; ++i, ++item_no) {
            const WorkItem it = p.work[i];
            const int L = p.seq_lens[it.b];
            const int t0 = it.t0, t1 = it.t1;
            const int nt = (t1 - t0 + kTile - 1) / kTile;
            const int last_vis = L - p.q_len + (row_valid ? row_seq / p.s.H : 0);
            float base = -CUDART_INF_F, l = 0.f;   // running base (log2 units), this half's row-sum share
            bool bad_item = false;
            for (int t = 0; t < nt && ok; ++t, ++T) {
                bad_item |= block_of(p, it.b, t0 / kTile + t) < 0;
                if (owned(T)) {
                    const int k = T >> 1;
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full, k & 1, bars, p.status))) { ok = false; break; }
                    tc_fence_after();
                    uint32_t sv[32];
                    if (tid == 64) PTRACE(5, T);
                    TMEM_LD32(lane_addr + kColS + 32 * hs, sv);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&bars->s_free);
                    const int tile_start = t0 + t * kTile + 32 * hs;
                    const int n_vis = row_valid ? max(0, min(t1, last_vis + 1) - tile_start) : 0;
                    // scores stay unscaled where the scale is positive: the row max then
                    // commutes with the scaling and each exponent argument is one fma
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
                    {
                        float other = -CUDART_INF_F;
                        if (!__all_sync(0xffffffffu, exchange(mx, other))) { ok = false; break; }
                        mx = fmaxf(mx, other);
                    }
                    if (tid == 64) PTRACE(6, T);
                    float alpha = 1.f;
                    bool rescale = false;
                    const float m_new = fmaxf(base, mx);
                    if (m_new > base + 8.f) {
                        alpha = exp2f(base - m_new);      // 0 when nothing was accumulated yet
                        base = m_new;
                        rescale = t > 0;
                    }
                    // the new base goes to the other CTA right away (it continues the chain)
                    if (hs == 0) st_async_f32(peer_bbuf, base, peer_bmsg);
                    if (__any_sync(0xffffffffu, rescale) && !rescale_o(T - 1, alpha)) { ok = false; break; }
                    const float nmb = base == -CUDART_INF_F ? -CUDART_INF_F : -base;
                    float sum0 = 0.f, sum1 = 0.f;
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float a = ex2(fmaf(__uint_as_float(sv[2 * j]), cs, nmb));
                        const float c = ex2(fmaf(__uint_as_float(sv[2 * j + 1]), cs, nmb));
                        const __nv_bfloat162 hh = __floats2bfloat162_rn(a, c);
                        pk[j] = *(const uint32_t *)&hh;
                        sum0 += a;           // fp32 row sum: the LSE does not see the rounding of P
                        sum1 += c;
                    }
                    l = l * alpha + (sum0 + sum1);
                    // this CTA's P buffer T % 2 is free once both PVs of tile T-2 are done:
                    // its own, and the other CTA's, whose completion also means the copy
                    // out of this buffer has finished reading it
                    if (k >= 1) {
                        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[T & 1], ((T >> 1) - 1) & 1, bars, p.status) &&
                                                         mbar_wait(&bars->rbuf_free, (k - 1) & 1, bars, p.status))) {
                            ok = false;
                            break;
                        }
                    }
                    if (tid == 64) PTRACE(7, T);
                    // P into this CTA's buffer and, by 16-byte remote stores that complete
                    // on the other CTA's p_rx barrier, into the other CTA's buffer
                    const uint32_t pofs = (T & 1) * kPBytes;
                    uint8_t *pbuf = smem + kOffP + pofs;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const uint4 v = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                        const uint32_t o = sw128(row, 4 * hs + ch);
                        *(uint4 *)(pbuf + o) = v;
                        st_async_v4(peer_pbase + pofs + o, v, peer_prx);
                    }
                    ++n_own_sent;
                    fence_proxy_async();
                    tc_fence_before();
                    mbar_arrive(&bars->ready[T & 1]);
                    if (tid == 64) PTRACE(10, T);
                } else {
                    // a tile the other CTA owns: its base (the chain), then the rescale
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars->bmsg, (T >> 1) & 1, bars, p.status))) { ok = false; break; }
                    const float b_new = *(volatile float *)(bbuf + row);
                    if (tid == 64) PTRACE(9, T);
                    if (tid == 64) mbar_expect_tx(&bars->bmsg, kRows * 4);    // arm the next message's phase
                    float alpha = 1.f;
                    bool rescale = false;
                    if (b_new > base) {
                        alpha = exp2f(base - b_new);
                        rescale = t > 0;
                        base = b_new;
                    }
                    if (__any_sync(0xffffffffu, rescale) && !rescale_o(T - 1, alpha)) { ok = false; break; }
                    l *= alpha;
                    // ready[T % 2] may run at most one phase ahead of the MMA thread: PV(T-2)
                    // has completed before tile T is declared ready (owned tiles wait for it
                    // anyway, before reusing their P buffer)
                    if (T >= 2 &&
                        !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[T & 1], ((T >> 1) - 1) & 1, bars, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_before();
                    mbar_arrive(&bars->ready[T & 1]);
                    if (tid == 64) PTRACE(10, T);
                }
            }
            // ---- end of this item: stage the next item's tensor-memory Q while the last
            // PV runs, swap row sums, write this item's output through the Q region, then
            // load the next item's shared-memory Q part.
            const bool have_next = i + 1 < i1 && has_own_tile(i + 1, T);
            if (ok && have_next) ok = __all_sync(0xffffffffu, issue_q(i + 1, 0));
            if (ok && nt > 0) {
                const int tl = T - 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->pv_done[tl & 1], (tl >> 1) & 1, bars, p.status));
            }
            float l_other = 0.f;
            if (ok) ok = __all_sync(0xffffffffu, exchange(l, l_other));
            float l_row = l + l_other;
            // the other CTA's share of the row sums
            const int lb = item_no & 1;
            if (ok && hs == 0)
                st_async_f32(mapa(smem_u32(lbuf + lb * 128 + row), peer), l_row, mapa(smem_u32(&bars->lmsg[lb]), peer));
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->lmsg[lb], (item_no >> 1) & 1, bars, p.status));
            if (ok) {
                l_row += *(volatile float *)(lbuf + lb * 128 + row);
                if (tid == 64) mbar_expect_tx(&bars->lmsg[lb], kRows * 4);
            }
            tc_fence_after();
            if (ok && have_next) ok = load_q_tmem(i + 1);
            if (ok && have_next)
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->qreg_free, (uses - 1) & 1, bars, p.status));
            const bool bad = aborted(bars) || !ok || bad_item;
            if (ok) {
                const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
                const uint64_t keep = l2_policy_evict_last();
                uint8_t *box = smem + kOffQ + (warp - 2) * kEpiBoxBytes;
                const int y = g * kRows + 32 * wq;
                const bool store = y < rows_seq;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    if (c > 0) {                       // the previous box was read
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
                    }
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t ov[32];
                        TMEM_LD32(lane_addr + kColO + 128 * hs + 64 * c + 32 * hh, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t pk[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(ov[8 * q + 2 * e]) * inv,
                                                                                __uint_as_float(ov[8 * q + 2 * e + 1]) * inv);
                                pk[e] = *(const uint32_t *)&h2;
                            }
                            *(uint4 *)(box + sw128(lane, 4 * hh + q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0 && store) {
                        tma_store_3d_hint(&o_map, box, 256 * (int)h + 128 * hs + 64 * c, y, i, keep);
                        bulk_commit();
                    }
                }
                if (lane == 0) bulk_wait_read();
                __syncwarp();
            }
            mbar_arrive(&bars->qreg_free);
            ++uses;
            if (row_valid && h == 0 && hs == 0)
                p.part_lse[(size_t)i * rows_seq + row_seq] =
                    bad ? CUDART_NAN_F : (l_row > 0.f ? base + log2f(l_row) : -CUDART_INF_F);
            tc_fence_before();     // O reads complete before the next item's first PV
            if (ok && have_next) ok = __all_sync(0xffffffffu, issue_q(i + 1, kQRounds));
        }
        if (lane == 0) bulk_wait_all();   // this warp's output stores have landed
        // the other CTA's PV of this CTA's last tile: its completion arrives here
        if (ok && n_own_sent > 0) mbar_wait(&bars->rbuf_free, (n_own_sent - 1) & 1, bars, p.status);
    }
    tc_fence_before();
    __syncthreads();
    // no message or copy of either CTA is still addressed to the other
    cluster_sync();
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

static void fill_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, dim3 grid, cudaStream_t st) {
    cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
}

}  // namespace pair

// Pairs that can be resident at once on the current device (0 if unknown).
int pair_max_clusters() {
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] > 0) return cached[dev];
    if (cudaFuncSetAttribute(pair::decode_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pair::kSmemBytes) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair::fill_config(cfg, attr, dim3(2, 1, 1), 0);
    cfg.numAttrs = 1;                        // cluster shape only
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair::decode_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached[dev] = n;
    return n;
}

cudaError_t launch_decode_pair(const DecodeParams &p, int32_t max_work, cudaStream_t st) {
    pair::PairParams pp;
    pp.p = p;
    pp.row_tiles = (p.q_len * p.s.H + pair::kRows - 1) / pair::kRows;
    CUtensorMap kv_map, q_map, o_map;
    if (!pair::make_map(&kv_map, p.latent, (uint64_t)p.s.num_blocks * p.s.bs, pair::kTile, (uint64_t)p.s.E()))
        return cudaErrorInvalidValue;
    const int rows_seq = p.q_len * p.s.H;
    if (!pair::make_map(&q_map, p.q, (uint64_t)p.B * rows_seq, pair::kRows, pair::kD)) return cudaErrorInvalidValue;
    if (!pair::make_out_map(&o_map, p.part_o, p.s.r, rows_seq, max_work)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(pair::decode_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pair::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair::fill_config(cfg, attr, dim3(2, pp.row_tiles, p.streams), st);
    return cudaLaunchKernelEx(&cfg, pair::decode_pair_kernel, kv_map, q_map, o_map, pp);
}

}  // namespace mla

#ifdef MLA_TRACE
extern "C" int mla_pair_trace_read(long long *events, long long *starts) {
    cudaError_t e = cudaMemcpyFromSymbol(events, mla::pair::g_ptrace, sizeof(mla::pair::g_ptrace));
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(starts, mla::pair::g_pstart, sizeof(mla::pair::g_pstart));
    return (int)e;
}
#endif
