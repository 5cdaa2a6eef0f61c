// The two rotations of the rotated-INT2 cache on the tensor cores, kv_lora_rank 512:
//   q_rot[m, :] = q_lat[m, :] . R          (query prep, before attention): qrot_kernel,
//                                          below, with R split into two bf16 halves
//   o_lat[m, :] = o_rot[m, :] . R^T        (after the split merge, before W_UV, when the
//                                          up-projection is not folded): rot_gemm_kernel
// rot_gemm_kernel computes Y[M x 512] = X[M x 512] . op(R), op = identity or
// transpose. R is first converted per call to fp16 (R16); the GEMM's B tiles come
// from R16 by TMA, the A tiles (fp32 merged outputs) are converted to fp16 by the
// threads that stage them in shared memory, and the MMA accumulates in fp32 in
// tensor memory. A CTA computes a [128 x 128] tile of Y over eight 64-wide K chunks:
// warps 1..7 convert the whole A tile into shared memory chunk by chunk (one chunk of
// loads in flight ahead), while warp 0 streams B through four stages and issues each
// chunk's MMAs as soon as its A and B are there.
//
// Also here: the merge of split partials into one latent row per (sequence,
// draft position, head), which precedes the second rotation.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

#include <cudaTypedefs.h>
#include <math_constants.h>
#include <string.h>

namespace mla {
namespace rot {

using namespace ptx;

constexpr int kThreads = 256;                   // warp 0: TMA + MMA issue; warps 1..7 convert A
constexpr int kConvThreads = kThreads - 32;
constexpr int kK = 512;                         // kv_lora_rank
constexpr int kTm = 128, kTn = 128, kKc = 64;   // tile M, tile N, K chunk
constexpr int kChunks = kK / kKc;               // 8
constexpr int kBStages = 4;
constexpr uint32_t kABytes = kTm * 128;         // one chunk of A: [128 rows x 64 k] fp16
constexpr uint32_t kBBytes = kTn * 128;         // one chunk of B: [128 j x 64 k] fp16 (either layout)
constexpr uint32_t kOffA = 0;                   // all of A: 8 chunks, 128 KB
constexpr uint32_t kOffB = kChunks * kABytes;   // kBStages B stages, 64 KB
constexpr uint32_t kOffBar = kOffB + kBStages * kBBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr unsigned long long kTimeoutNs = 2000000000ull;
constexpr int kJobsPerConv = (kTm * 8 + kConvThreads - 1) / kConvThreads;   // 16-byte A chunks per thread

struct RotParams {
    const void *X;
    int ldx;              // elements per X row
    void *Y;
    int ldy;              // elements per Y row
    int M;
    int copy_rope;        // > 0: copy X[:, 512 : 512 + copy_rope] (bf16) to Y as fp16
    int32_t *status;
};

__device__ __forceinline__ uint4 pack8_f16(const float *v) {
    const __half2 h0 = __floats2half2_rn(v[0], v[1]);
    const __half2 h1 = __floats2half2_rn(v[2], v[3]);
    const __half2 h2 = __floats2half2_rn(v[4], v[5]);
    const __half2 h3 = __floats2half2_rn(v[6], v[7]);
    return make_uint4(*(const uint32_t *)&h0, *(const uint32_t *)&h1, *(const uint32_t *)&h2, *(const uint32_t *)&h3);
}

// Y[m, 512 + d] = fp16(X[m, 512 + d]) for the copy_rope dims of part `part` of `nparts`
// row ranges of rows m0 .. m0 + 127 (bf16 X): 16-byte vectors.
__device__ __forceinline__ void copy_rope_f16(const RotParams &rp, int m0, int tid, int nthreads, int part,
                                              int nparts) {
    if (rp.copy_rope <= 0) return;
    const int vec = rp.copy_rope / 8;            // 8-element vectors per row
    const int rows = (kTm + nparts - 1) / nparts;
    const int r0 = part * rows;
    const int total = rows * vec;
#pragma unroll 4
    for (int job = tid; job < total; job += nthreads) {
        const int r = r0 + job / vec, c = job % vec, m = m0 + r;
        if (r >= kTm || m >= rp.M) continue;
        const uint4 u = __ldg((const uint4 *)((const __nv_bfloat16 *)rp.X + (size_t)m * rp.ldx + kK) + c);
        const __nv_bfloat162 *hv = (const __nv_bfloat162 *)&u;
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(hv[e]);
            f[2 * e] = x.x;
            f[2 * e + 1] = x.y;
        }
        *((uint4 *)((__half *)rp.Y + (size_t)m * rp.ldy + kK) + c) = pack8_f16(f);
    }
}

// R16 = fp16(R), round to nearest even, eight elements per thread.
__global__ void __launch_bounds__(256) r_to_f16_kernel(const float *R, __half *R16, int n8) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
        const float4 a = ((const float4 *)R)[2 * i], b = ((const float4 *)R)[2 * i + 1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        ((uint4 *)R16)[i] = pack8_f16(v);
    }
}

// X_FP32: X is fp32 (else bf16). TRANS: op(R) = R^T (else R). Y_F16: Y is fp16 (else fp32).
// r_map: R16 as [512 rows, 512 cols] fp16, 128B-swizzled boxes of [64 cols x 128
// rows] (TRANS: B = R rows j, K-major) or [64 cols x 64 rows] (else: B = R rows k,
// MN-major, two 64-wide j atoms per chunk).
template <bool X_FP32, bool TRANS, bool Y_F16>
__global__ void __launch_bounds__(kThreads, 1) rot_gemm_kernel(const __grid_constant__ CUtensorMap r_map,
                                                               const RotParams rp) {
    const int m0 = blockIdx.x * kTm, j0 = blockIdx.y * kTn;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *a_full = (uint64_t *)(smem + kOffBar);     // [kChunks] A chunk converted
    uint64_t *b_full = a_full + kChunks;                 // [kBStages] B tile landed
    uint64_t *b_free = b_full + kBStages;                // [kBStages] MMAs reading the stage done
    uint64_t *mma_fin = b_free + kBStages;
    uint32_t *tmem_slot = (uint32_t *)(mma_fin + 1);
    int32_t *abort_flag = (int32_t *)(mma_fin + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < kChunks; ++i) mbar_init(&a_full[i], kConvThreads);
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_free[i], 1);
        }
        mbar_init(mma_fin, 1);
        abort_flag[0] = 0;
        abort_flag[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTn)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    if (warp == 0) {
        if (lane == 0) {
            // fp16 A and B, fp32 D, M 128, N 128; B MN-major for op(R) = R (R's rows are k)
            const uint32_t idesc = (1u << 4) | ((TRANS ? 0u : 1u) << 16) | ((uint32_t)(kTn >> 3) << 17) |
                                   ((uint32_t)(kTm >> 4) << 24);
            int last_b[kBStages];
            auto issue_b = [&](int kc) {     // TMA of chunk kc's B tile into stage kc % kBStages
                const int st = kc % kBStages;
                uint8_t *Bm = smem + kOffB + st * kBBytes;
                last_b[st] = kc;
                mbar_expect_tx(&b_full[st], kBBytes);
                if (TRANS) {
                    tma_load_2d(Bm, &r_map, kc * kKc, j0, &b_full[st]);
                } else {
                    for (int atom = 0; atom < kTn / 64; ++atom)
                        tma_load_2d(Bm + atom * (kKc * 128), &r_map, j0 + 64 * atom, kc * kKc, &b_full[st]);
                }
            };
            for (int st = 0; st < kBStages; ++st) {
                last_b[st] = -1;
                if (st < kChunks) issue_b(st);
            }
            bool ok = true;
            for (int kc = 0; kc < kChunks && ok; ++kc) {
                const int st = kc % kBStages;
                ok = mbar_wait_bounded(&a_full[kc], 0, abort_flag, rp.status, FLAG_TIMEOUT, kTimeoutNs) &&
                     mbar_wait_bounded(&b_full[st], (kc / kBStages) & 1, abort_flag, rp.status, FLAG_TIMEOUT,
                                       kTimeoutNs);
                if (!ok) break;
                tc_fence_after();
                const uint64_t a0 = sdesc(smem_u32(smem + kOffA + kc * kABytes), 16, 1024);
                const uint8_t *Bm = smem + kOffB + st * kBBytes;
                const uint64_t b0 = TRANS ? sdesc(smem_u32(Bm), 16, 1024) : sdesc(smem_u32(Bm), kKc * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < kKc / 16; ++kk) {
                    const uint64_t bd = b0 + (uint64_t)((TRANS ? 32 * kk : 2048 * kk) >> 4);
                    mma_ss(tmem, a0 + (uint64_t)((32 * kk) >> 4), bd, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&b_free[st]);
                if (kc + kBStages < kChunks) {      // refill the stage once its MMAs are done
                    ok = mbar_wait_bounded(&b_free[st], (kc / kBStages) & 1, abort_flag, rp.status, FLAG_TIMEOUT,
                                           kTimeoutNs);
                    if (ok) issue_b(kc + kBStages);
                }
            }
            mma_commit(mma_fin);
            if (!ok) {
                // never leave a B copy in flight into this CTA's shared memory: a stage's
                // earlier copies landed before its later one was issued, so waiting for
                // the last one of each stage is enough (bounded, regardless of the abort)
                for (int st = 0; st < kBStages; ++st)
                    if (last_b[st] >= 0)
                        mbar_wait_bounded(&b_full[st], (last_b[st] / kBStages) & 1, abort_flag + 1, nullptr, 0,
                                          kTimeoutNs);
            }
        }
        __syncwarp();
    } else {
        // A: rows m0.., k = 64 kc + 8 ch .. +7 -> fp16, K-major swizzled; the next
        // chunk's loads are issued before this chunk is converted and stored
        const int ct = tid - 32;
        uint4 ra[kJobsPerConv][2], rb[kJobsPerConv][2];
        auto load = [&](int kc, uint4 (&r)[kJobsPerConv][2]) {
#pragma unroll
            for (int i = 0; i < kJobsPerConv; ++i) {
                const int job = ct + kConvThreads * i, row = job >> 3, ch = job & 7, m = m0 + row;
                r[i][0] = make_uint4(0, 0, 0, 0);
                r[i][1] = make_uint4(0, 0, 0, 0);
                if (job < kTm * 8 && m < rp.M) {
                    const size_t base = (size_t)m * rp.ldx + kc * kKc + 8 * ch;
                    if (X_FP32) {
                        r[i][0] = *(const uint4 *)((const float *)rp.X + base);
                        r[i][1] = *(const uint4 *)((const float *)rp.X + base + 4);
                    } else {
                        r[i][0] = *(const uint4 *)((const __nv_bfloat16 *)rp.X + base);
                    }
                }
            }
        };
        auto store = [&](int kc, const uint4 (&r)[kJobsPerConv][2]) {
            uint8_t *A = smem + kOffA + kc * kABytes;
#pragma unroll
            for (int i = 0; i < kJobsPerConv; ++i) {
                const int job = ct + kConvThreads * i, row = job >> 3, ch = job & 7;
                if (job >= kTm * 8) continue;
                float v[8];
                if (X_FP32) {
                    const float *f0 = (const float *)&r[i][0], *f1 = (const float *)&r[i][1];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[e] = f0[e];
                        v[4 + e] = f1[e];
                    }
                } else {
                    const __nv_bfloat162 *h = (const __nv_bfloat162 *)&r[i][0];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h[e]);
                        v[2 * e] = f.x;
                        v[2 * e + 1] = f.y;
                    }
                }
                *(uint4 *)(A + sw128(row, ch)) = pack8_f16(v);
            }
            fence_proxy_async();
            mbar_arrive(&a_full[kc]);
        };
        load(0, ra);
        for (int kc = 0; kc < kChunks; kc += 2) {
            load(kc + 1, rb);
            store(kc, ra);
            if (kc + 2 < kChunks) load(kc + 2, ra);
            store(kc + 1, rb);
        }
    }
    // everyone: the MMAs are done (or the CTA gave up)
    bool ok = mbar_wait_bounded(mma_fin, 0, abort_flag, rp.status, FLAG_TIMEOUT, kTimeoutNs) &&
              *(volatile int32_t *)abort_flag == 0;
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (warp < 4) {
        const int m = m0 + 32 * warp + lane;
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
        for (int c = 0; c < kTn / 32; ++c) {
            uint32_t v[32];
            if (ok) {
                TMEM_LD32(taddr + 32 * c, v);
                tmem_wait_ld();
            }
            if (m >= rp.M) continue;
            const int j = j0 + 32 * c;
            if (Y_F16) {
                __half *dst = (__half *)rp.Y + (size_t)m * rp.ldy + j;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = ok ? __uint_as_float(v[8 * q + e]) : CUDART_NAN_F;
                    *(uint4 *)(dst + 8 * q) = pack8_f16(f);
                }
            } else {
                float *dst = (float *)rp.Y + (size_t)m * rp.ldy + j;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float4 f;
                    f.x = ok ? __uint_as_float(v[4 * q + 0]) : CUDART_NAN_F;
                    f.y = ok ? __uint_as_float(v[4 * q + 1]) : CUDART_NAN_F;
                    f.z = ok ? __uint_as_float(v[4 * q + 2]) : CUDART_NAN_F;
                    f.w = ok ? __uint_as_float(v[4 * q + 3]) : CUDART_NAN_F;
                    *(float4 *)(dst + 4 * q) = f;
                }
            }
        }
    }
    // the query's rope part passes through unrotated (bf16 -> fp16)
    if (blockIdx.y == 0) copy_rope_f16(rp, m0, tid, kThreads, 0, 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTn) : "memory");
    }
}

// ---- the query rotation, q_rot = q_lat . R, without converting the query --------
// R is split into two bf16 matrices, R = R_hi + R_lo + e with R_hi = bf16(R) and R_lo
// = bf16(R - R_hi) (|e| <= 2^-17 |R|, finer than one fp16 rounding of R), so that the
// bf16 query rows feed the tensor cores straight from TMA: per K-step two MMAs (with
// R_hi and with R_lo) accumulate into the same fp32 tile. A CTA computes a [128 x 128]
// tile of q_rot over eight 64-wide K chunks in four TMA stages (A: [128 rows x 64 k]
// query box; B: [64 k x 128 j] of R_hi and of R_lo, MN-major); lane 0 of warp 0
// issues the copies and the MMAs, four warps read the tile out as fp16.
constexpr int kQThreads = 128;
constexpr int kQStages = 4;
constexpr uint32_t kQStageBytes = kABytes + 2 * kBBytes;          // 48 KB
constexpr uint32_t kQOffBar = kQStages * kQStageBytes;            // 192 KB
constexpr uint32_t kQSmemBytes = kQOffBar + 256 + 1024;

__global__ void __launch_bounds__(256) r_split_bf16_kernel(const float *R, __nv_bfloat16 *Rhi, __nv_bfloat16 *Rlo, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float v = R[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        Rhi[i] = hi;
        Rlo[i] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
}

__global__ void __launch_bounds__(kQThreads, 1) qrot_kernel(const __grid_constant__ CUtensorMap q_map,
                                                            const __grid_constant__ CUtensorMap rhi_map,
                                                            const __grid_constant__ CUtensorMap rlo_map,
                                                            const RotParams rp) {
    const int m0 = blockIdx.x * kTm, j0 = blockIdx.y * kTn;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + kQOffBar);      // [kQStages] chunk landed
    uint64_t *freed = full + kQStages;                   // [kQStages] MMAs reading the stage done
    uint64_t *mma_fin = freed + kQStages;
    uint32_t *tmem_slot = (uint32_t *)(mma_fin + 1);
    int32_t *abort_flag = (int32_t *)(mma_fin + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();
    if (tid == 0) {
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&freed[i], 1);
        }
        mbar_init(mma_fin, 1);
        abort_flag[0] = 0;
        abort_flag[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTn)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    if (warp == 0 && lane == 0) {
        // bf16 A and B, fp32 D, M 128, N 128, B MN-major (R's rows are k)
        constexpr uint32_t idesc = idesc_bf16(kTm, kTn, true);
        int last[kQStages];
        auto issue = [&](int kc) {           // chunk kc's A and B boxes into stage kc % kQStages
            const int st = kc % kQStages;
            uint8_t *S = smem + st * kQStageBytes;
            last[st] = kc;
            mbar_expect_tx(&full[st], kQStageBytes);
            tma_load_2d(S, &q_map, kc * kKc, m0, &full[st]);
            for (int atom = 0; atom < kTn / 64; ++atom) {
                tma_load_2d(S + kABytes + atom * (kKc * 128), &rhi_map, j0 + 64 * atom, kc * kKc, &full[st]);
                tma_load_2d(S + kABytes + kBBytes + atom * (kKc * 128), &rlo_map, j0 + 64 * atom, kc * kKc, &full[st]);
            }
        };
        for (int st = 0; st < kQStages; ++st) {
            last[st] = -1;
            if (st < kChunks) issue(st);
        }
        bool ok = true;
        for (int kc = 0; kc < kChunks && ok; ++kc) {
            const int st = kc % kQStages;
            ok = mbar_wait_bounded(&full[st], (kc / kQStages) & 1, abort_flag, rp.status, FLAG_TIMEOUT, kTimeoutNs);
            if (!ok) break;
            tc_fence_after();
            const uint8_t *S = smem + st * kQStageBytes;
            const uint64_t a0 = sdesc(smem_u32(S), 16, 1024);
            const uint64_t bh = sdesc(smem_u32(S + kABytes), kKc * 128, 1024);
            const uint64_t bl = sdesc(smem_u32(S + kABytes + kBBytes), kKc * 128, 1024);
#pragma unroll
            for (int kk = 0; kk < kKc / 16; ++kk) {
                const uint64_t a = a0 + (uint64_t)((32 * kk) >> 4);
                mma_ss(tmem, a, bh + (uint64_t)((2048 * kk) >> 4), idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                mma_ss(tmem, a, bl + (uint64_t)((2048 * kk) >> 4), idesc, 1u);
            }
            mma_commit(&freed[st]);
            if (kc + kQStages < kChunks) {      // refill the stage once its MMAs are done
                ok = mbar_wait_bounded(&freed[st], (kc / kQStages) & 1, abort_flag, rp.status, FLAG_TIMEOUT, kTimeoutNs);
                if (ok) issue(kc + kQStages);
            }
        }
        mma_commit(mma_fin);
        if (!ok) {
            // never leave a copy in flight into this CTA's shared memory (bounded waits)
            for (int st = 0; st < kQStages; ++st)
                if (last[st] >= 0)
                    mbar_wait_bounded(&full[st], (last[st] / kQStages) & 1, abort_flag + 1, nullptr, 0, kTimeoutNs);
        }
    }
    __syncwarp();
    bool ok = mbar_wait_bounded(mma_fin, 0, abort_flag, rp.status, FLAG_TIMEOUT, kTimeoutNs) &&
              *(volatile int32_t *)abort_flag == 0;
    ok = __syncthreads_and(ok);
    tc_fence_after();
    // Epilogue: the fp32 tile -> fp16 rows staged in shared memory (the stages are free:
    // every MMA has completed and every copy into them landed), then stored as whole
    // 256-byte row segments; rows 272 bytes apart, so that a warp's staging writes fall
    // on distinct banks.
    constexpr int kRowB = kTn * 2 + 16;
    uint8_t *stg = smem;
    {
        const int r = 32 * warp + lane;
        const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
        for (int c = 0; c < kTn / 32; ++c) {
            uint32_t v[32];
            if (ok) {
                TMEM_LD32(taddr + 32 * c, v);
                tmem_wait_ld();
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = ok ? __uint_as_float(v[8 * q + e]) : CUDART_NAN_F;
                *(uint4 *)(stg + r * kRowB + (32 * c + 8 * q) * 2) = pack8_f16(f);
            }
        }
    }
    __syncthreads();
    constexpr int kVecs = kTn / 8;                  // 16-byte vectors a row segment
    for (int idx = tid; idx < kTm * kVecs; idx += kQThreads) {
        const int r = idx / kVecs, cv = idx % kVecs, m = m0 + r;
        if (m < rp.M)
            *((uint4 *)((__half *)rp.Y + (size_t)m * rp.ldy + j0) + cv) = *(const uint4 *)(stg + r * kRowB + 16 * cv);
    }
    // the query's rope part passes through unrotated (bf16 -> fp16), a quarter of the
    // rows by each of the row tile's column-tile CTAs
    copy_rope_f16(rp, m0, tid, kQThreads, blockIdx.y, gridDim.y);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTn) : "memory");
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

template <bool X_FP32, bool TRANS, bool Y_F16>
static cudaError_t launch_t(const __half *R16, const RotParams &rp, cudaStream_t st) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    CUtensorMap map;
    memset(&map, 0, sizeof map);
    cuuint64_t dims[2] = {(cuuint64_t)kK, (cuuint64_t)kK};
    cuuint64_t strides[1] = {(cuuint64_t)kK * 2};
    cuuint32_t box[2] = {64, TRANS ? (cuuint32_t)kTn : 64u};
    cuuint32_t estr[2] = {1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(R16), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(rot_gemm_kernel<X_FP32, TRANS, Y_F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((rp.M + kTm - 1) / kTm, kK / kTn);
    return launch_pdl(rot_gemm_kernel<X_FP32, TRANS, Y_F16>, grid, dim3(kThreads), kSmemBytes, st, map, rp);
}

// Merge the split partials of each (b, i, h) row into o_rot[(b * q_len + i) * H + h]
// and its log2-sum-exp; write an identity schedule (sequence b -> slot b) so
// that the up-projection reads the merged rows as one-split partials.
__global__ void __launch_bounds__(256) merge_rows_kernel(CombineParams c, float *o_rot, float *lse2, int32_t *ident) {
    const int H = c.s.H, rows_seq = c.q_len * H;
    const int total = c.B * rows_seq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0)
        for (int b = threadIdx.x; b <= c.B; b += blockDim.x) ident[b] = b;
    for (int rowg = blockIdx.x * 8 + warp; rowg < total; rowg += gridDim.x * 8) {
        const int b = rowg / rows_seq, row = rowg % rows_seq;
        const int s0 = c.split_start[b], s1 = c.split_start[b + 1];
        bool nan = s1 <= s0;
        float M = -CUDART_INF_F;
        for (int s = s0; s < s1; ++s) {
            const float v = c.part_lse[(size_t)s * rows_seq + row];
            nan |= isnan(v);
            M = fmaxf(M, v);
        }
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.f;
        float tot = 0.f;
        for (int s = s0; s < s1; ++s) {
            const float v = c.part_lse[(size_t)s * rows_seq + row];
            const float w = v == -CUDART_INF_F ? 0.f : exp2f(v - M);
            tot += w;
            const size_t at = ((size_t)s * rows_seq + row) * kK;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = c.part_bf16 ? bf16x4_to_float4(((const uint2 *)((const __nv_bfloat16 *)c.part_o + at))[lane + 32 * q])
                                             : ((const float4 *)((const float *)c.part_o + at))[lane + 32 * q];
                acc[4 * q + 0] = fmaf(w, f.x, acc[4 * q + 0]);
                acc[4 * q + 1] = fmaf(w, f.y, acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(w, f.z, acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(w, f.w, acc[4 * q + 3]);
            }
        }
        const float inv = tot > 0.f ? 1.f / tot : 0.f;
        float4 *dst = (float4 *)(o_rot + (size_t)rowg * kK);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float4 f;
            f.x = nan ? CUDART_NAN_F : acc[4 * q + 0] * inv;
            f.y = nan ? CUDART_NAN_F : acc[4 * q + 1] * inv;
            f.z = nan ? CUDART_NAN_F : acc[4 * q + 2] * inv;
            f.w = nan ? CUDART_NAN_F : acc[4 * q + 3] * inv;
            dst[lane + 32 * q] = f;
        }
        if (lane == 0) lse2[rowg] = nan ? CUDART_NAN_F : M + log2f(tot);
    }
}

}  // namespace rot

bool rot_tc_supported(const ShapeArgs &s) { return s.r == rot::kK; }

cudaError_t launch_rot_query(const float *R, __nv_bfloat16 *Rsplit, const void *q_bf16, void *q_rot_f16, int rows,
                             int D, int32_t *status, cudaStream_t st, bool split_done) {
    const int n = rot::kK * rot::kK;
    __nv_bfloat16 *Rhi = Rsplit, *Rlo = Rsplit + n;
    cudaError_t e = cudaSuccess;
    if (!split_done) {               // (the planner's launch usually splits R already)
        rot::r_split_bf16_kernel<<<(n + 255) / 256, 256, 0, st>>>(R, Rhi, Rlo, n);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto fn = rot::encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    CUtensorMap qm, hm, lm;
    memset(&qm, 0, sizeof qm);
    cuuint32_t estr[2] = {1, 1};
    {   // the query rows [rows, D] bf16: boxes of [64 k x 128 rows], rows past the end read 0
        cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)rot::kTm};
        if (fn(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q_bf16), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    for (int which = 0; which < 2; ++which) {   // R_hi, R_lo [512 k, 512 j] bf16: boxes of [64 j x 64 k]
        cuuint64_t dims[2] = {(cuuint64_t)rot::kK, (cuuint64_t)rot::kK};
        cuuint64_t strides[1] = {(cuuint64_t)rot::kK * 2};
        cuuint32_t box[2] = {64, 64};
        if (fn(which ? &lm : &hm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, which ? (void *)Rlo : (void *)Rhi, dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    rot::RotParams rp;
    rp.X = q_bf16;
    rp.ldx = D;
    rp.Y = q_rot_f16;
    rp.ldy = D;
    rp.M = rows;
    rp.copy_rope = D - rot::kK;
    rp.status = status;
    e = cudaFuncSetAttribute(rot::qrot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rot::kQSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((rows + rot::kTm - 1) / rot::kTm, rot::kK / rot::kTn);
    return launch_pdl(rot::qrot_kernel, grid, dim3(rot::kQThreads), rot::kQSmemBytes, st, qm, hm, lm, rp);
}

cudaError_t launch_rot_output(const CombineParams &c, __half *R16, float *o_rot, float *o_lat, float *lse2,
                              int32_t *ident, int32_t *status, cudaStream_t st) {
    const int rows = c.B * c.q_len * c.s.H;
    const int n8 = rot::kK * rot::kK / 8;
    rot::r_to_f16_kernel<<<(n8 + 255) / 256, 256, 0, st>>>(c.R, R16, n8);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
    rot::merge_rows_kernel<<<min((rows + 7) / 8, 4096), 256, 0, st>>>(c, o_rot, lse2, ident);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    rot::RotParams rp;
    rp.X = o_rot;
    rp.ldx = rot::kK;
    rp.Y = o_lat;
    rp.ldy = rot::kK;
    rp.M = rows;
    rp.copy_rope = 0;
    rp.status = status;
    return rot::launch_t<true, true, false>(R16, rp, st);
}

}  // namespace mla
