// Split combine + W_UV up-projection on the tensor cores (bf16 cache kind,
// kv_lora_rank 512, v_head_dim 128).
//
// One CTA per (head h, tile of up to 64 output rows), a row being a (sequence,
// draft position) pair. TMA streams W_UV^h ([512 x 128] bf16, 128 KB) into shared
// memory from the CTA's start, while the decode kernel is still finishing; once the
// partials are complete, the threads merge each row's split partials (bf16 or fp32) by their
// log2-sum-exp into the latent output o_lat (fp32 accumulate, stored bf16 as a
// K-major 128B-swizzled operand) and write the row's LSE. One thread then
// issues 32 tcgen05 MMAs, D[128 x NR] = W_UV^hT [128 x 512] . o_lat^T [512 x NR]
// (A = W_UV^h read MN-major straight from its row-major layout), and four warps
// read D out of tensor memory and store out[b, i, h, :] in bf16.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

#include <cudaTypedefs.h>
#include <math_constants.h>
#include <string.h>

namespace mla {
namespace comb {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kR = 512, kDv = 128;
constexpr int kMaxRows = 64;                        // output rows per CTA (MMA N)
constexpr uint32_t kWBoxBytes = 64 * 128;            // [64 k x 64 v] bf16
constexpr uint32_t kWBytes = kR * kDv * 2;           // 128 KB
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffO = kWBytes;                  // o_lat: 8 column blocks of [kMaxRows x 128 B]
constexpr uint32_t kOBlockBytes = kMaxRows * 128;
constexpr uint32_t kOffBar = kOffO + 8 * kOBlockBytes;
constexpr int kWarps = kThreads / 32;
// rows with many splits, few rows: each warp's partial merge of its share of a row's
// splits (max, sum, 512 unnormalised dims), merged once more per row
constexpr uint32_t kOffPart = kOffBar + 64 + 8 * kMaxRows;
constexpr uint32_t kPartBytes = kWarps * (8 + kR * 4);
constexpr uint32_t kSmemBytes = kOffPart + kPartBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr unsigned long long kTimeoutNs = 2000000000ull;

struct CombTcParams {
    CombineParams c;
    int32_t rows;          // B * q_len
};

// Phase timestamps (globaltimer) per CTA for performance analysis, compiled only
// with -DMLA_TRACE: entry, after the grid dependency wait, partials merged, W_UV
// landed, MMAs done, end. Product builds contain none of it.
#ifdef MLA_TRACE
__device__ unsigned long long g_comb_time[1024][6];
#define COMB_TRACE(slot)                                                                      \
    do {                                                                                      \
        const unsigned cid = blockIdx.y * gridDim.x + blockIdx.x;                             \
        if (threadIdx.x == 0 && cid < 1024) g_comb_time[cid][slot] = globaltimer();            \
    } while (0)
#else
#define COMB_TRACE(slot) \
    do {                 \
    } while (0)
#endif

__global__ void __launch_bounds__(kThreads, 1)
combine_tc_kernel(const __grid_constant__ CUtensorMap w_map, const CombTcParams tp) {
    const CombineParams &c = tp.c;
    const int h = blockIdx.x;
    const int row0 = blockIdx.y * kMaxRows;
    const int nrows = min(kMaxRows, tp.rows - row0);
    const int NR = (nrows + 15) & ~15;               // MMA N: multiple of 16
    const int H = c.s.H, rows_seq = c.q_len * H;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bar_w = (uint64_t *)(smem + kOffBar);
    uint64_t *bar_mma = bar_w + 1;
    uint32_t *tmem_slot = (uint32_t *)(bar_w + 2);
    int32_t *abort_flag = (int32_t *)(bar_w + 3);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    COMB_TRACE(0);

    // Set-up that overlaps the decode kernel's tail: barriers, TMEM, and the TMA of
    // W_UV^h ([512 x 128] bf16) into shared memory. W_UV is an input no kernel of this
    // call writes, and the planner lets the kernels after it launch only once every
    // earlier kernel of the stream has completed, so it may be read before the wait.
    if (tid == 0) {
        mbar_init(bar_w, 1);
        mbar_init(bar_mma, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
        mbar_expect_tx(bar_w, kWBytes);
        for (int vb = 0; vb < 2; ++vb)
            for (int kb = 0; kb < 8; ++kb)
                tma_load_2d(smem + kOffW + (vb * 8 + kb) * kWBoxBytes, &w_map, 64 * vb, h * kR + 64 * kb, bar_w);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(64)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // ---- merge split partials: warp per row, each lane owns 16 latent dims. Every
    // row's split range is read first (before the dependency wait when the planner
    // that wrote them is known to have completed); then a row costs one round trip:
    // its log2-sum-exps and partials (up to four splits at a time) are loaded together
    // and merged with a running maximum.
    int2 *s_range = (int2 *)(smem + kOffBar + 64);   // [kMaxRows] split ranges
    auto read_ranges = [&]() {
        if (tid < nrows) {
            const int b = (row0 + tid) / c.q_len;
            s_range[tid] = make_int2(c.split_start[b], c.split_start[b + 1]);
        }
    };
    if (c.ranges_early) read_ranges();
    pdl_wait();                      // the split partials are complete from here on
    COMB_TRACE(1);
    if (!c.ranges_early) read_ranges();
    __syncthreads();
    // Rows of 8 or fewer: each row's splits are dealt to wpr = 16 / rows warps (split
    // sb + wpr k to warp sub of the row), each merging its share; the row's warp then
    // merges the wpr partials. More rows: one warp per row merges all of its splits.
    const int wpr = nrows <= kWarps / 2 ? kWarps / nrows : 1;
    // one split batch (up to four splits, stride `step`) merged into (M, tot, acc)
    auto merge_splits = [&](int row, int s_first, int s_end, int step, float &M, float &tot, float (&acc)[16],
                            bool &nan) {
        for (int sb = s_first; sb < s_end; sb += 4 * step) {
            float4 f[4][4];
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int sp = sb + k * step;
                v[k] = -CUDART_INF_F;
                if (sp < s_end) {
                    const size_t at = ((size_t)sp * rows_seq + row) * kR;
                    if (c.part_bf16) {      // 4 bf16 per (lane, q): half the bytes of fp32
                        const uint2 *po = (const uint2 *)((const __nv_bfloat16 *)c.part_o + at);
#pragma unroll
                        for (int q = 0; q < 4; ++q) f[k][q] = bf16x4_to_float4(po[lane + 32 * q]);
                    } else {
                        const float4 *po = (const float4 *)((const float *)c.part_o + at);
#pragma unroll
                        for (int q = 0; q < 4; ++q) f[k][q] = po[lane + 32 * q];
                    }
                    v[k] = c.part_lse[(size_t)sp * rows_seq + row];
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) f[k][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            float Mn = M;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                nan |= isnan(v[k]);
                Mn = fmaxf(Mn, v[k]);
            }
            // rescale what was merged so far (nothing, or the earlier splits)
            const float a = M == -CUDART_INF_F ? 0.f : exp2f(M - Mn);
            tot *= a;
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] *= a;
            M = Mn;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float wgt = v[k] == -CUDART_INF_F ? 0.f : exp2f(v[k] - M);
                tot += wgt;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[4 * q + 0] = fmaf(wgt, f[k][q].x, acc[4 * q + 0]);
                    acc[4 * q + 1] = fmaf(wgt, f[k][q].y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(wgt, f[k][q].z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(wgt, f[k][q].w, acc[4 * q + 3]);
                }
            }
        }
    };
    float *part_ms = (float *)(smem + kOffPart);                  // [kWarps][2]: M, tot
    float *part_acc = (float *)(smem + kOffPart + 8 * kWarps);    // [kWarps][kR]
    int *part_nan = (int *)(smem + kOffBar + 48);                 // rows whose splits hold a NaN
    if (wpr > 1) {
        if (tid == 0) *part_nan = 0;
        __syncthreads();
        const int rr = warp / wpr, sub = warp % wpr;
        float M = -CUDART_INF_F, tot = 0.f, acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;
        bool nan = false;
        if (rr < nrows) {
            const int2 sr = s_range[rr];
            const int row = ((row0 + rr) % c.q_len) * H + h;
            merge_splits(row, sr.x + sub, sr.y, wpr, M, tot, acc, nan);
        }
        if (lane == 0) {
            part_ms[2 * warp] = M;
            part_ms[2 * warp + 1] = tot;
            if (nan) atomicOr(part_nan, 1 << rr);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *(float4 *)(part_acc + warp * kR + 4 * (lane + 32 * q)) =
                make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        __syncthreads();
    }
    for (int rr = warp; rr < NR; rr += kWarps) {
        const int grow = row0 + rr;
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;
        float lse_out = 0.f;
        if (rr < nrows) {
            const int i = grow % c.q_len;
            const int2 sr = s_range[rr];
            const int row = i * H + h;
            bool nan = sr.y <= sr.x;
            float M = -CUDART_INF_F, tot = 0.f;
            if (wpr == 1) {
                merge_splits(row, sr.x, sr.y, 1, M, tot, acc, nan);
            } else {
                // the row's wpr partials, each weighted by 2^(M_j - M)
                nan |= ((*part_nan >> rr) & 1) != 0;
                for (int j = 0; j < wpr; ++j) M = fmaxf(M, part_ms[2 * (rr * wpr + j)]);
                for (int j = 0; j < wpr; ++j) {
                    const int w = rr * wpr + j;
                    const float Mj = part_ms[2 * w];
                    const float wgt = Mj == -CUDART_INF_F ? 0.f : exp2f(Mj - M);
                    tot = fmaf(wgt, part_ms[2 * w + 1], tot);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 a = *(const float4 *)(part_acc + w * kR + 4 * (lane + 32 * q));
                        acc[4 * q + 0] = fmaf(wgt, a.x, acc[4 * q + 0]);
                        acc[4 * q + 1] = fmaf(wgt, a.y, acc[4 * q + 1]);
                        acc[4 * q + 2] = fmaf(wgt, a.z, acc[4 * q + 2]);
                        acc[4 * q + 3] = fmaf(wgt, a.w, acc[4 * q + 3]);
                    }
                }
            }
            const float inv = tot > 0.f ? 1.f / tot : 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] = nan ? CUDART_NAN_F : acc[k] * inv;
            lse_out = nan ? CUDART_NAN_F : (M + log2f(tot)) * kLn2;
            if (lane == 0) c.lse[(size_t)grow * H + h] = lse_out;
        }
        // dims d = 4*(lane + 32q) .. +3 -> column block d/64, chunk (d%64)/8, half (d%8)/4
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int d = 4 * (lane + 32 * q);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[4 * q + 0], acc[4 * q + 1]);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[4 * q + 2], acc[4 * q + 3]);
            uint2 u;
            u.x = *(const uint32_t *)&lo;
            u.y = *(const uint32_t *)&hi;
            uint8_t *blk = smem + kOffO + (d >> 6) * kOBlockBytes;
            *(uint2 *)(blk + sw128(rr, (d & 63) >> 3) + ((d & 7) >> 2) * 8) = u;
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    COMB_TRACE(2);
    const uint32_t tmem = *tmem_slot;

    if (tid == 0) {
        bool ok = mbar_wait_bounded(bar_w, 0, abort_flag, nullptr, 0, kTimeoutNs);
        COMB_TRACE(3);
        if (ok) {
            tc_fence_after();
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(NR >> 3) << 17) |
                                   ((uint32_t)(128 >> 4) << 24);
            const uint64_t a0 = sdesc(smem_u32(smem + kOffW), 8 * kWBoxBytes, 1024);   // MN-major W
            const uint64_t b0 = sdesc(smem_u32(smem + kOffO), 16, 1024);               // K-major o_lat
            for (int j = 0; j < kR / 16; ++j) {
                const int kb = j >> 2, ks = j & 3;
                const uint64_t a = a0 + (uint64_t)((kb * kWBoxBytes + ks * 2048) >> 4);
                const uint64_t bd = b0 + (uint64_t)((kb * kOBlockBytes + ks * 32) >> 4);
                mma_ss(tmem, a, bd, idesc, j > 0 ? 1u : 0u);
            }
        }
        mma_commit(bar_mma);
    }
    __syncwarp();
    if (warp < 4) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_mma, 0, abort_flag, nullptr, 0, kTimeoutNs));
        COMB_TRACE(4);
        tc_fence_after();
        const int v = 32 * warp + lane;              // TMEM lane = output dim
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
        __nv_bfloat16 *out = (__nv_bfloat16 *)c.out;
        for (int cb = 0; cb < NR; cb += 32) {
            uint32_t vals[32];
            if (ok) {
                TMEM_LD32(taddr + cb, vals);
                tmem_wait_ld();
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int rr = cb + k;
                if (rr < nrows) {
                    const float f = ok ? __uint_as_float(vals[k]) : CUDART_NAN_F;
                    out[((size_t)(row0 + rr) * H + h) * kDv + v] = __float2bfloat16_rn(f);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    COMB_TRACE(5);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64) : "memory");
    }
}

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

}  // namespace comb

bool combine_tc_supported(const ShapeArgs &s) {
    return (s.kind == MLA_KV_BF16 || is_int2(s.kind)) && s.r == comb::kR && s.dv == comb::kDv;
}

cudaError_t launch_combine_tc(const CombineParams &c, cudaStream_t st) {
    auto fn = comb::encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    CUtensorMap map;
    memset(&map, 0, sizeof map);
    // W_UV as [H * r rows (k), d_v cols (v)], boxes of [64 k x 64 v]
    cuuint64_t dims[2] = {(cuuint64_t)comb::kDv, (cuuint64_t)c.s.H * comb::kR};
    cuuint64_t strides[1] = {(cuuint64_t)comb::kDv * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(c.W_UV), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    comb::CombTcParams tp;
    tp.c = c;
    tp.rows = c.B * c.q_len;
    cudaError_t e = cudaFuncSetAttribute(comb::combine_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)comb::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(c.s.H, (tp.rows + comb::kMaxRows - 1) / comb::kMaxRows);
    return launch_pdl(comb::combine_tc_kernel, grid, dim3(comb::kThreads), comb::kSmemBytes, st, map, tp);
}

}  // namespace mla

#ifdef MLA_TRACE
extern "C" int mla_comb_trace_read(unsigned long long *host, int n) {
    return (int)cudaMemcpyFromSymbol(host, mla::comb::g_comb_time, sizeof(unsigned long long) * 6 * (size_t)n);
}
#endif
