// CUDA-core kernels of the library: the split-KV planner, the append /
// quantise path, the query rotation, the generic decode and the split combine
// with the W_UV up-projection.
//
// The generic decode handles every supported shape and cache kind; the
// tensor-core decode (mla_tc.cu) replaces it for the DeepSeek-V3-shaped bf16
// and INT2 caches. Both write the same partial format, so the planner and the
// combine here serve both.
#include "mla_internal.cuh"

#include <math_constants.h>

#include <algorithm>

namespace mla {

// ============================================================================
// Planner. The cache of every valid sequence is cut into units of plan_tile tokens
// (64: one cache block; 128: the two blocks the bf16 tensor-core kernel scores per
// MMA); each sequence is also charged item_cost units for its start. The
// concatenation of all sequences' costs is split into `streams` contiguous runs of
// equal cost. A work item is the intersection of one sequence with one run, so
// every stream gets the same cost (the last unit of a sequence may be short) and
// the schedule has at most streams + B items. Items are listed sequence by
// sequence, which also lists them stream by stream. One CTA; the schedule lives
// in the workspace, so no launch needs the lengths on the host.
// ============================================================================
constexpr int kPlanTile = 64;      // plan_tile when the caller leaves it 0

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, at
// most 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int *s_warp, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
        int w = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        s_warp[lane] = w - x;          // exclusive warp offsets
        if (lane == 31) s_warp[32] = w;
    }
    __syncthreads();
    const int excl = s_warp[warp] + incl - v;
    total = s_warp[32];
    __syncthreads();
    return excl;
}

#ifdef MLA_TRACE
// planner timestamps (globaltimer): entry, after the grid dependency wait, end
__device__ unsigned long long g_plan_time[3];
__device__ __forceinline__ unsigned long long ptx_globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
extern "C" int mla_plan_trace_read(unsigned long long *host) {
    return (int)cudaMemcpyFromSymbol(host, g_plan_time, sizeof g_plan_time);
}
#endif
__device__ __forceinline__ void plan_body(const DecodeParams &p, int32_t max_work) {
    __shared__ int s_warp[33];
    __shared__ long long s_tiles;
    // per sequence slot of the current chunk (dynamic shared memory, blockDim slots):
    // cost position of the first tile, first stream, first item (chunk-local), tiles,
    // length
    extern __shared__ long long plan_slots[];
    long long *s_tb = plan_slots, *s_first = plan_slots + blockDim.x;
    int *s_loc = (int *)(plan_slots + 2 * blockDim.x), *s_n = s_loc + blockDim.x, *s_len = s_n + blockDim.x;
#ifdef MLA_TRACE
    if (threadIdx.x == 0) g_plan_time[0] = ptx_globaltimer();
#endif
    // Wait first, then let the decode kernel launch: everything after the planner
    // (which may start work before its own wait, e.g. loading W_UV) then starts only
    // once every kernel before the planner has completed.
    pdl_wait();
    pdl_trigger();
#ifdef MLA_TRACE
    if (threadIdx.x == 0) g_plan_time[1] = ptx_globaltimer();
#endif
    const int tid = threadIdx.x;
    const int64_t cap = (int64_t)p.max_blocks * p.s.bs;
    const int P = p.streams;
    if (tid == 0) { s_tiles = 0; p.status[0] = 0; }
    __syncthreads();
    // Cost axis: each sequence is charged item_cost units for its start (the query
    // load and epilogue of a new work item) followed by one unit per tile; streams
    // take equal cost ranges, so a stream that starts more sequences gets fewer tiles.
    const int ic = p.item_cost;
    const int PT = p.plan_tile > 0 ? p.plan_tile : kPlanTile;
    long long local = 0;
    for (int b = tid; b < p.B; b += blockDim.x) {
        const int L = p.seq_lens[b];
        if (L >= p.q_len && L <= cap) local += (L + PT - 1) / PT + ic;
        else raise_flag(p.status, FLAG_BAD_LENGTH);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if ((tid & 31) == 0) atomicAdd((unsigned long long *)&s_tiles, (unsigned long long)local);   // one per warp
    __syncthreads();
    const long long NC = s_tiles;
    const long long T = NC > 0 ? (NC + P - 1) / P : 1;      // cost per stream
    int tile_carry = 0, item_carry = 0;
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int n = 0, L = 0;
        if (b < p.B) {
            L = p.seq_lens[b];
            if (L >= p.q_len && L <= cap) n = (L + PT - 1) / PT;
        }
        int tot_tiles, tot_items;
        // tb: cost position of the sequence's first tile (after its start charge)
        const long long tb = tile_carry + block_exclusive_scan(n > 0 ? n + ic : 0, s_warp, tot_tiles) + ic;
        const long long first = tb / T;
        const long long last = n > 0 ? (tb + n - 1) / T : first - 1;
        const int cnt = (int)(last - first + 1);
        const int loc = block_exclusive_scan(cnt, s_warp, tot_items);   // first item, within this chunk
        if (b < p.B) ((int32_t *)p.split_start)[b] = item_carry + loc;
        // One item of sequence slot i: the work item (within max_work) and
        // stream_start[s] = index of the first item whose stream is >= s, for the
        // item's own stream and, for a sequence's first item, also the streams from
        // the one after the stream holding the cost position just before the
        // sequence's start charge.
        auto write_item = [&](int slot, int k, int idx, long long tbi, long long first_i, int ni, int Li) {
            const long long sgi = first_i + k;
            if (idx < max_work) {
                const long long lo = (sgi * T > tbi ? sgi * T : tbi) - tbi;
                const long long hi = ((sgi + 1) * T < tbi + ni ? (sgi + 1) * T : tbi + ni) - tbi;
                WorkItem it;
                it.b = base + slot;
                it.t0 = (int)(lo * PT);
                it.t1 = (int)min((long long)Li, hi * PT);
                it.stream = (int)sgi;
                ((WorkItem *)p.work)[idx] = it;
            }
            long long s_lo = sgi;
            if (k == 0) {
                const long long cb = tbi - ic;
                s_lo = cb > 0 ? (cb - 1) / T + 1 : 0;
            }
            for (long long st = s_lo; st <= sgi && st < P; ++st) ((int32_t *)p.stream_start)[st] = min(idx, max_work);
        };
        // a thread writes its own sequence's items unless some sequence has many (the
        // per-item path below pays a search and a barrier: measured slower for a
        // DeepSeek-V3 batch of 32 sequences of up to 6 items, faster for two sequences
        // of about 38)
        if (!__syncthreads_or(cnt > 12)) {
            if (b < p.B) {
                const int start = item_carry + loc;
                for (int k = 0; k < cnt && start + k < max_work; ++k) {
                    const long long sg = first + k;
                    const long long lo = (sg * T > tb ? sg * T : tb) - tb;
                    const long long hi = ((sg + 1) * T < tb + n ? (sg + 1) * T : tb + n) - tb;
                    WorkItem it;
                    it.b = b;
                    it.t0 = (int)(lo * PT);
                    it.t1 = (int)min((long long)L, hi * PT);
                    it.stream = (int)sg;
                    ((WorkItem *)p.work)[start + k] = it;
                }
                if (n > 0) {
                    const long long cb = tb - ic;
                    const long long prev = cb > 0 ? (cb - 1) / T : -1;
                    for (long long st = prev + 1; st <= last && st < P; ++st)
                        ((int32_t *)p.stream_start)[st] = min(start + (int)(st > first ? st - first : 0), max_work);
                }
            }
        } else {
            // many (a few long sequences): the chunk's items one per thread; item j
            // belongs to the last slot whose first item is <= j (slots without items
            // share the next one's start)
            s_loc[tid] = loc;
            s_tb[tid] = tb;
            s_first[tid] = first;
            s_n[tid] = n;
            s_len[tid] = L;
            __syncthreads();
            for (int j = tid; j < tot_items; j += blockDim.x) {
                int lo_i = 0, hi_i = blockDim.x - 1;
                while (lo_i < hi_i) {
                    const int mid = (lo_i + hi_i + 1) >> 1;
                    if (s_loc[mid] <= j) lo_i = mid;
                    else hi_i = mid - 1;
                }
                write_item(lo_i, j - s_loc[lo_i], item_carry + j, s_tb[lo_i], s_first[lo_i], s_n[lo_i], s_len[lo_i]);
            }
        }
        __syncthreads();                     // the slots are rewritten by the next chunk
        tile_carry += tot_tiles;
        item_carry += tot_items;
    }
    const int total = min(item_carry, max_work);
    if (tid == 0) {
        ((int32_t *)p.split_start)[p.B] = item_carry;
        ((int32_t *)p.num_work)[0] = total;
    }
    // streams past the last sequence's last stream, and the end marker stream_start[P]
    for (long long st = (NC > 0 ? (NC - 1) / T : -1) + 1 + tid; st <= P; st += blockDim.x)
        ((int32_t *)p.stream_start)[st] = total;
#ifdef MLA_TRACE
    __syncthreads();
    if (tid == 0) g_plan_time[2] = ptx_globaltimer();
#endif
}

__global__ void __launch_bounds__(1024) plan_kernel(DecodeParams p, int32_t max_work) { plan_body(p, max_work); }

cudaError_t launch_plan(const DecodeParams &p, int32_t max_work, cudaStream_t st) {
    // one thread per sequence (whole warps, at most 1024): fewer threads, cheaper barriers
    const int threads = p.B >= 1024 ? 1024 : ((p.B + 31) / 32) * 32;
    const int nt = threads > 0 ? threads : 32;
    return launch_pdl(plan_kernel, dim3(1), dim3(nt), (size_t)nt * 28, st, p, max_work);
}

// ============================================================================
// Query rotation for the rotated-INT2 cache: q_prep[row] = [q_lat . R ; q_R],
// fp32 accumulation. 32 query rows per CTA, each thread owns NC output dims.
// ============================================================================
// OUT: 0 fp32 (CUDA-core decode), 1 fp16 (tensor-core decode of the INT2 cache).
template <int NC, int OUT>
__global__ void __launch_bounds__(256) qprep_kernel(DecodeParams p, const float *R, void *q_prep, int rows) {
    extern __shared__ float sq[];                 // [32][RD]
    const int RD = p.s.RD(), D = p.s.D();         // rotated dims (r, or all D for INT2_JOINT)
    const int row0 = blockIdx.x * 32;
    const __nv_bfloat16 *q = (const __nv_bfloat16 *)p.q;
    for (int idx = threadIdx.x; idx < 32 * RD; idx += blockDim.x) {
        int rr = idx / RD, k = idx % RD, row = row0 + rr;
        sq[idx] = row < rows ? __bfloat162float(q[(size_t)row * D + k]) : 0.f;
    }
    __syncthreads();
    float acc[32][NC];
#pragma unroll
    for (int rr = 0; rr < 32; ++rr)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[rr][c] = 0.f;
    for (int k = 0; k < RD; ++k) {
        float Rk[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            int j = threadIdx.x + 256 * c;
            Rk[c] = j < RD ? __ldg(R + (size_t)k * RD + j) : 0.f;
        }
#pragma unroll
        for (int rr = 0; rr < 32; ++rr) {
            float qv = sq[rr * RD + k];
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[rr][c] = fmaf(qv, Rk[c], acc[rr][c]);
        }
    }
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
        int row = row0 + rr;
        if (row >= rows) break;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            int j = threadIdx.x + 256 * c;
            if (j < RD) {
                if (OUT == 1) ((__half *)q_prep)[(size_t)row * D + j] = __float2half_rn(acc[rr][c]);
                else ((float *)q_prep)[(size_t)row * D + j] = acc[rr][c];
            }
        }
        // the dims outside the rotation (the rope part, unless INT2_JOINT) as given
        for (int j = RD + threadIdx.x; j < D; j += blockDim.x) {
            const float v = __bfloat162float(q[(size_t)row * D + j]);
            if (OUT == 1) ((__half *)q_prep)[(size_t)row * D + j] = __float2half_rn(v);
            else ((float *)q_prep)[(size_t)row * D + j] = v;
        }
    }
}

template <int OUT>
static cudaError_t launch_qprep_t(const DecodeParams &p, const float *R, void *q_prep, cudaStream_t st) {
    const int rows = p.B * p.q_len * p.s.H;
    const int RD = p.s.RD();
    const size_t smem = (size_t)32 * RD * sizeof(float);
    dim3 grid((rows + 31) / 32);
    if (RD <= 256) {
        cudaFuncSetAttribute(qprep_kernel<1, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        qprep_kernel<1, OUT><<<grid, 256, smem, st>>>(p, R, q_prep, rows);
    } else if (RD <= 512) {
        cudaFuncSetAttribute(qprep_kernel<2, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        qprep_kernel<2, OUT><<<grid, 256, smem, st>>>(p, R, q_prep, rows);
    } else if (RD <= 768) {
        cudaFuncSetAttribute(qprep_kernel<3, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        qprep_kernel<3, OUT><<<grid, 256, smem, st>>>(p, R, q_prep, rows);
    } else {
        cudaFuncSetAttribute(qprep_kernel<4, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        qprep_kernel<4, OUT><<<grid, 256, smem, st>>>(p, R, q_prep, rows);
    }
    return cudaGetLastError();
}

// A query that comes in the rotated basis: bf16 -> the decode kernels' operand type,
// 8 elements (16 bytes in) per thread step.
template <int OUT>
__global__ void __launch_bounds__(256) convert_query_kernel(const __nv_bfloat16 *q, void *out, size_t n8) {
    pdl_trigger();
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 u = ((const uint4 *)q)[i];
        const __nv_bfloat162 *h = (const __nv_bfloat162 *)&u;
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(h[e]);
            f[2 * e] = x.x;
            f[2 * e + 1] = x.y;
        }
        if (OUT == 1) {
            __half2 o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
            ((uint4 *)out)[i] = *(const uint4 *)o;
        } else {
            ((float4 *)out)[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
            ((float4 *)out)[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
}

cudaError_t launch_convert_query(const void *q, void *out, size_t n, bool out_f16, cudaStream_t st) {
    const size_t n8 = n / 8;                      // n = rows * (r + d_R), a multiple of 8
    const int blocks = (int)std::min<size_t>((n8 + 255) / 256, 2048);
    return out_f16 ? launch_pdl(convert_query_kernel<1>, dim3(blocks), dim3(256), 0, st, (const __nv_bfloat16 *)q, out, n8)
                   : launch_pdl(convert_query_kernel<0>, dim3(blocks), dim3(256), 0, st, (const __nv_bfloat16 *)q, out, n8);
}

cudaError_t launch_qprep(const DecodeParams &p, const float *R, void *q_prep, bool out_f16, cudaStream_t st) {
    return out_f16 ? launch_qprep_t<1>(p, R, q_prep, st) : launch_qprep_t<0>(p, R, q_prep, st);
}

// ============================================================================
// Generic split-KV decode. One CTA = one work item x 16 query rows (a row is a
// (draft position i, head h) pair). Per 32-token tile: gather the tile through
// the block table into shared memory as fp32 (dequantising INT2), scores with
// one lane per token, online softmax per row in log2 units, then P.C into
// per-thread accumulators (thread owns latent dims tid + 256c for all rows).
// Output: normalised partial latent output and its log2-sum-exp per row.
// ============================================================================
constexpr int kRB = 16;   // query rows per CTA
constexpr int kTT = 32;   // tokens per tile

template <int KIND>
__device__ __forceinline__ void gather_tile(const DecodeParams &p, int b, int tb, int t1, float *sK,
                                            int Dp, int *sValid) {
    const int D = p.s.D(), r = p.s.r, dR = p.s.dR, bs = p.s.bs;
    if (threadIdx.x < kTT) {
        int t = tb + threadIdx.x;
        int ok = 0;
        if (t < t1) {
            int lb = t / bs;
            int blk = lb < p.max_blocks ? p.block_table[(size_t)b * p.max_blocks + lb] : -1;
            if (blk >= 0 && blk < p.s.num_blocks) ok = 1 + blk;   // store blk+1
            else raise_flag(p.status, FLAG_BAD_BLOCK);
        }
        sValid[threadIdx.x] = ok;
    }
    __syncthreads();
    if (KIND == MLA_KV_BF16) {
        const int nvec = D / 8;                       // 16-byte chunks per token row
        for (int idx = threadIdx.x; idx < kTT * nvec; idx += blockDim.x) {
            int tt = idx / nvec, v = idx % nvec;
            int blk1 = sValid[tt];
            float *dst = sK + tt * Dp + v * 8;
            if (blk1) {
                size_t row = (size_t)(blk1 - 1) * bs + (tb + tt) % bs;
                uint4 u = *((const uint4 *)((const __nv_bfloat16 *)p.latent + row * p.s.E()) + v);
                const __nv_bfloat16 *h = (const __nv_bfloat16 *)&u;
#pragma unroll
                for (int e = 0; e < 8; ++e) dst[e] = __bfloat162float(h[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) dst[e] = 0.f;
            }
        }
    } else if (KIND == MLA_KV_FP32) {
        const int nvec = D / 4;
        for (int idx = threadIdx.x; idx < kTT * nvec; idx += blockDim.x) {
            int tt = idx / nvec, v = idx % nvec;
            int blk1 = sValid[tt];
            float *dst = sK + tt * Dp + v * 4;
            if (blk1) {
                size_t row = (size_t)(blk1 - 1) * bs + (tb + tt) % bs;
                float4 u = *((const float4 *)((const float *)p.latent + row * p.s.E()) + v);
                dst[0] = u.x; dst[1] = u.y; dst[2] = u.z; dst[3] = u.w;
            } else {
                dst[0] = dst[1] = dst[2] = dst[3] = 0.f;
            }
        }
    } else {
        // INT2: one thread per code byte (4 dims), then the bf16 rope key (INT2_ROT_QR:
        // the rope key's codes follow the latent's in the row, so the bytes cover it).
        const int nbytes = p.s.QD() / 4, gs = p.s.gs, ng = p.s.QD() / gs;
        for (int idx = threadIdx.x; idx < kTT * nbytes; idx += blockDim.x) {
            int tt = idx / nbytes, k = idx % nbytes;
            int blk1 = sValid[tt];
            float *dst = sK + tt * Dp + 4 * k;
            if (blk1) {
                size_t row = (size_t)(blk1 - 1) * bs + (tb + tt) % bs;
                unsigned byte = p.codes[row * nbytes + k];
                int g = (4 * k) / gs;
                float sc = __half2float(p.scale_zero[(row * ng + g) * 2 + 0]);
                float zr = __half2float(p.scale_zero[(row * ng + g) * 2 + 1]);
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = __fmaf_rn((float)((byte >> (2 * e)) & 3u), sc, zr);
            } else {
                dst[0] = dst[1] = dst[2] = dst[3] = 0.f;
            }
        }
        if (p.s.kind == MLA_KV_INT2_ROT) {
            for (int idx = threadIdx.x; idx < kTT * dR; idx += blockDim.x) {
                int tt = idx / dR, d = idx % dR;
                int blk1 = sValid[tt];
                float v = 0.f;
                if (blk1) {
                    size_t row = (size_t)(blk1 - 1) * bs + (tb + tt) % bs;
                    v = __bfloat162float(p.rope[row * dR + d]);
                }
                sK[tt * Dp + r + d] = v;
            }
        }
    }
}

template <int KIND, int NC>
__global__ void __launch_bounds__(256) decode_simt_kernel(DecodeParams p) {
    const int w = blockIdx.x;
    if (w >= p.num_work[0]) return;
    const WorkItem item = p.work[w];
    const int b = item.b, t0 = item.t0, t1 = item.t1, slot = w;
    const int H = p.s.H, D = p.s.D(), Dp = D + 1;
    const int r = p.s.OD();               // dims of the latent-space output (INT2_JOINT: all D)
    const int rows_total = p.q_len * H;
    const int row0 = blockIdx.y * kRB;
    if (row0 >= rows_total) return;
    const int L = p.seq_lens[b];

    extern __shared__ float smem[];
    float *sQ = smem;                     // [kRB][D]
    float *sK = sQ + kRB * D;             // [kTT][Dp]
    float *sP = sK + kTT * Dp;            // [kRB][kTT]
    float *sA = sP + kRB * kTT;           // [kRB] rescale factors
    float *sL = sA + kRB;                 // [kRB]
    float *sM = sL + kRB;                 // [kRB]
    int *sValid = (int *)(sM + kRB);      // [kTT]
    __shared__ int s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_bad = 0;
    for (int idx = tid; idx < kRB * D; idx += blockDim.x) {
        int rr = idx / D, d = idx % D, row = row0 + rr;
        float v = 0.f;
        if (row < rows_total) {
            size_t off = ((size_t)b * rows_total + row) * D + d;   // q is [B][q_len][H][D]
            if (KIND == MLA_KV_INT2_ROT) v = p.q_prep[off];
            else if (KIND == MLA_KV_FP32) v = ((const float *)p.q)[off];
            else v = __bfloat162float(((const __nv_bfloat16 *)p.q)[off]);
        }
        sQ[idx] = v;
    }

    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.f, 0.f};
    int last_vis[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        int row = row0 + warp + 8 * j;
        last_vis[j] = row < rows_total ? (L - p.q_len + row / H) : -1;
    }
    float acc[kRB][NC];
#pragma unroll
    for (int rr = 0; rr < kRB; ++rr)
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[rr][c] = 0.f;

    for (int tb = t0; tb < t1; tb += kTT) {
        __syncthreads();                  // previous tile fully consumed
        gather_tile<KIND>(p, b, tb, t1, sK, Dp, sValid);
        __syncthreads();
        if (tid < kTT && tb + tid < t1 && !sValid[tid]) s_bad = 1;
        float sc[2];
        {
            // both rows of this warp against the lane's token, 4 independent chains
            const float *q0 = sQ + warp * D, *q1 = sQ + (warp + 8) * D, *kr = sK + lane * Dp;
            float a0 = 0.f, a1 = 0.f, c0 = 0.f, c1 = 0.f;
            for (int d = 0; d < D; d += 2) {
                const float k0 = kr[d], k1 = kr[d + 1];
                a0 = fmaf(q0[d], k0, a0);
                a1 = fmaf(q0[d + 1], k1, a1);
                c0 = fmaf(q1[d], k0, c0);
                c1 = fmaf(q1[d + 1], k1, c1);
            }
            sc[0] = a0 + a1;
            sc[1] = c0 + c1;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int rr = warp + 8 * j;
            const float s = sc[j];
            const int t = tb + lane;
            const bool vis = (t < t1) && (t <= last_vis[j]) && sValid[lane];
            const float s2 = vis ? s * p.scale_log2 : -CUDART_INF_F;
            const float m_new = fmaxf(m_run[j], warp_max(s2));
            const float pr = vis ? exp2f(s2 - m_new) : 0.f;
            const float alpha = (m_new == -CUDART_INF_F) ? 1.f : exp2f(m_run[j] - m_new);
            l_run[j] = l_run[j] * alpha + warp_sum(pr);
            m_run[j] = m_new;
            sP[rr * kTT + lane] = pr;
            if (lane == 0) sA[rr] = alpha;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < kRB; ++rr) {
            const float a = sA[rr];
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[rr][c] *= a;
        }
        const int ntok = min(kTT, t1 - tb);
        for (int tt = 0; tt < ntok; ++tt) {
            float kv[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                int d = tid + 256 * c;
                kv[c] = d < r ? sK[tt * Dp + d] : 0.f;
            }
#pragma unroll
            for (int rr = 0; rr < kRB; ++rr) {
                const float pr = sP[rr * kTT + tt];
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[rr][c] = fmaf(pr, kv[c], acc[rr][c]);
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            sL[warp + 8 * j] = l_run[j];
            sM[warp + 8 * j] = m_run[j];
        }
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    for (int rr = 0; rr < kRB; ++rr) {
        const int row = row0 + rr;
        if (row >= rows_total) break;
        const float l = sL[rr];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *po = p.part_o + ((size_t)slot * rows_total + row) * r;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            int d = tid + 256 * c;
            if (d < r) po[d] = acc[rr][c] * inv;
        }
        if (tid == 0)
            p.part_lse[(size_t)slot * rows_total + row] =
                bad ? CUDART_NAN_F : (l > 0.f ? sM[rr] + log2f(l) : -CUDART_INF_F);
    }
}

template <int KIND>
static cudaError_t launch_decode_kind(const DecodeParams &p, int32_t max_work, cudaStream_t st) {
    const int D = p.s.D();
    const size_t smem = sizeof(float) * ((size_t)kRB * D + (size_t)kTT * (D + 1) + kRB * kTT + 3 * kRB) +
                        sizeof(int) * kTT;
    dim3 grid(max_work, (p.q_len * p.s.H + kRB - 1) / kRB);
    if (p.s.OD() <= 256) {
        cudaFuncSetAttribute(decode_simt_kernel<KIND, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        decode_simt_kernel<KIND, 1><<<grid, 256, smem, st>>>(p);
    } else if (p.s.OD() <= 512) {
        cudaFuncSetAttribute(decode_simt_kernel<KIND, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        decode_simt_kernel<KIND, 2><<<grid, 256, smem, st>>>(p);
    } else if (p.s.OD() <= 768) {
        cudaFuncSetAttribute(decode_simt_kernel<KIND, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        decode_simt_kernel<KIND, 3><<<grid, 256, smem, st>>>(p);
    } else {
        cudaFuncSetAttribute(decode_simt_kernel<KIND, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        decode_simt_kernel<KIND, 4><<<grid, 256, smem, st>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_simt(const DecodeParams &p, int32_t max_work, cudaStream_t st) {
    switch (p.s.kind) {
        case MLA_KV_BF16: return launch_decode_kind<MLA_KV_BF16>(p, max_work, st);
        case MLA_KV_FP32: return launch_decode_kind<MLA_KV_FP32>(p, max_work, st);
        default: return launch_decode_kind<MLA_KV_INT2_ROT>(p, max_work, st);
    }
}

// ============================================================================
// Combine: merge the split partials of each (b, i, h) row by their log2-sum-
// exp, rotate back (INT2: o_lat = o_rot . R^T) and up-project through W_UV^h.
// One CTA = one head x 8 rows (b, i), so W_UV^h is read once per 8 rows.
// ============================================================================
constexpr int kCR = 8;

template <bool FP32IO>
__global__ void __launch_bounds__(256) combine_kernel(CombineParams p) {
    extern __shared__ float cs[];
    const int H = p.s.H, r = p.s.r, dv = p.s.dv;
    const int od = p.s.OD();              // partial dims: r, or r + d_R (INT2_JOINT)
    const int h = blockIdx.x;
    const int nrows = p.B * p.q_len;
    const int rb0 = blockIdx.y * kCR;
    float *so = cs;                       // [kCR][od]
    float *st = so + kCR * od;            // [kCR][r] (INT2 rotation target)
    float *slse = st + kCR * r;           // [kCR]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows_total = p.q_len * H;

    // warp w merges row rb0 + w
    if (warp < kCR) {
        const int rb = rb0 + warp;
        float *dst = so + warp * od;
        if (rb < nrows) {
            const int b = rb / p.q_len, i = rb % p.q_len;
            const int s0 = p.split_start[b], s1 = p.split_start[b + 1];
            const int row = i * H + h;
            float M = -CUDART_INF_F;
            bool nan = (s1 <= s0);
            for (int s = s0; s < s1; ++s) {
                float v = p.part_lse[(size_t)s * rows_total + row];
                if (isnan(v)) nan = true;
                M = fmaxf(M, v);
            }
            float tot = 0.f;
            for (int s = s0; s < s1; ++s) {
                float v = p.part_lse[(size_t)s * rows_total + row];
                tot += (v == -CUDART_INF_F) ? 0.f : exp2f(v - M);
            }
            const float inv = tot > 0.f ? 1.f / tot : 0.f;
            for (int d = lane; d < od; d += 32) {
                float a = 0.f;
                for (int s = s0; s < s1; ++s) {
                    float v = p.part_lse[(size_t)s * rows_total + row];
                    float wgt = (v == -CUDART_INF_F) ? 0.f : exp2f(v - M) * inv;
                    const size_t at = ((size_t)s * rows_total + row) * od + d;
                    const float pv = p.part_bf16 ? __bfloat162float(((const __nv_bfloat16 *)p.part_o)[at])
                                                 : ((const float *)p.part_o)[at];
                    a = fmaf(wgt, pv, a);
                }
                dst[d] = nan ? CUDART_NAN_F : a;
            }
            if (lane == 0) slse[warp] = nan ? CUDART_NAN_F : (M + log2f(tot)) * kLn2;
        } else {
            for (int d = lane; d < od; d += 32) dst[d] = 0.f;
        }
    }
    __syncthreads();
    const float *src = so;
    if (p.R) {
        // o_lat[j] = sum_k R[j][k] o_rot[k] for j < r (R is [od, od]; INT2_JOINT keeps
        // the first r of the r + d_R rotated-back dims): a warp per (row, j), lanes over k.
        for (int job = warp; job < kCR * r; job += 8) {
            const int rr = job / r, j = job % r;
            const float *Rj = p.R + (size_t)j * od;
            float a = 0.f;
            for (int k = lane; k < od; k += 32) a = fmaf(__ldg(Rj + k), so[rr * od + k], a);
            a = warp_sum(a);
            if (lane == 0) st[rr * r + j] = a;
        }
        __syncthreads();
        src = st;
    }
    const int ss = p.R ? r : od;          // row stride of the up-projection's input
    // out[v] = sum_k o_lat[k] W_UV[h][k][v]; thread -> (v, k-phase)
    for (int v0 = 0; v0 < dv; v0 += 256) {
        const int v = v0 + tid;
        float a[kCR];
#pragma unroll
        for (int rr = 0; rr < kCR; ++rr) a[rr] = 0.f;
        if (v < dv) {
            for (int k = 0; k < r; ++k) {
                float wv;
                if (FP32IO) wv = __ldg((const float *)p.W_UV + ((size_t)h * r + k) * dv + v);
                else wv = __bfloat162float(((const __nv_bfloat16 *)p.W_UV)[((size_t)h * r + k) * dv + v]);
#pragma unroll
                for (int rr = 0; rr < kCR; ++rr) a[rr] = fmaf(src[rr * ss + k], wv, a[rr]);
            }
#pragma unroll
            for (int rr = 0; rr < kCR; ++rr) {
                const int rb = rb0 + rr;
                if (rb >= nrows) break;
                const size_t o = ((size_t)rb * H + h) * dv + v;
                const float val = isnan(slse[rr]) ? CUDART_NAN_F : a[rr];
                if (FP32IO) ((float *)p.out)[o] = val;
                else ((__nv_bfloat16 *)p.out)[o] = __float2bfloat16_rn(val);
            }
        }
    }
    if (tid < kCR) {
        const int rb = rb0 + tid;
        if (rb < nrows) p.lse[(size_t)rb * H + h] = slse[tid];
    }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((size_t)kCR * (p.s.OD() + p.s.r) + kCR);
    dim3 grid(p.s.H, (p.B * p.q_len + kCR - 1) / kCR);
    if (p.s.kind == MLA_KV_FP32) {
        cudaFuncSetAttribute(combine_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        combine_kernel<true><<<grid, 256, smem, st>>>(p);
    } else {
        cudaFuncSetAttribute(combine_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        combine_kernel<false><<<grid, 256, smem, st>>>(p);
    }
    return cudaGetLastError();
}

// ============================================================================
// Append. BF16 / FP32: one warp per new token, 16-byte vector copies of the
// latent and rope key into the token's slot. INT2: 16 tokens per CTA; rotation
// y = c . R as an fp32 fmaf chain over k ascending (the encoding definition's
// order, which fixes the integer codes), then per (token, group) clip, range,
// fp16 scale/zero, codes and 2-bit packing.
// ============================================================================
__device__ __forceinline__ int find_seq(const int32_t *cu_new, int B, int n) {
    int lo = 0, hi = B - 1;                   // largest b with cu_new[b] <= n
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu_new[mid] <= n) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Returns the token row index (blk * bs + slot) or -1 after raising a flag.
__device__ __forceinline__ long long locate_slot(const AppendParams &p, int n) {
    const int b = find_seq(p.cu_new, p.B, n);
    const int pos = p.start_pos[b] + (n - p.cu_new[b]);
    const int lb = pos / p.s.bs;
    if (pos < 0 || lb >= p.max_blocks) { raise_flag(p.status, FLAG_BAD_BLOCK); return -1; }
    const int blk = p.block_table[(size_t)b * p.max_blocks + lb];
    if (blk < 0 || blk >= p.s.num_blocks) { raise_flag(p.status, FLAG_BAD_BLOCK); return -1; }
    return (long long)blk * p.s.bs + pos % p.s.bs;
}

// New token n into its slot: one warp, 16-byte vectors.
template <typename T>
__device__ __forceinline__ void copy_token(const AppendParams &p, int n) {
    const int lane = threadIdx.x & 31;
    if (n >= p.num_new) return;
    long long row = 0;
    if (lane == 0) row = locate_slot(p, n);
    row = __shfl_sync(0xffffffffu, row, 0);
    if (row < 0) return;
    constexpr int E = 16 / sizeof(T);            // elements per 16-byte vector
    const int r = p.s.r, dR = p.s.dR;
    uint4 *dst = (uint4 *)((T *)p.latent + (size_t)row * p.s.E());
    const uint4 *src_c = (const uint4 *)((const T *)p.c_kv + (size_t)n * r);
    const uint4 *src_r = (const uint4 *)((const T *)p.k_rope + (size_t)n * dR);
    for (int v = lane; v < r / E; v += 32) dst[v] = src_c[v];
    for (int v = lane; v < dR / E; v += 32) dst[r / E + v] = src_r[v];
}

template <typename T>
__global__ void __launch_bounds__(256) append_copy_kernel(AppendParams p) {
    pdl_trigger();
    pdl_wait();
    copy_token<T>(p, blockIdx.x * 8 + (threadIdx.x >> 5));
}

// Work that needs no result of the planner, done by extra blocks of the planner's
// launch: the copy of a decode step's new tokens (bf16 / fp32 cache) and the split of
// the INT2 rotation R into bf16 halves for the query rotation.
struct PrepParams {
    AppendParams a;              // a.num_new == 0: no copy
    int32_t copy_blocks;         // blocks 1 .. copy_blocks copy tokens, a warp per token
    const float *R;              // nullptr: no split
    __nv_bfloat16 *Rhi, *Rlo;
    int32_t r_n;                 // elements of R
};

// The decode's planner (block 0), then the copy blocks, then the R-split blocks. Every
// block waits for the previous kernel of the stream first, as separate kernels would.
template <typename T>
__global__ void __launch_bounds__(1024) plan_prep_kernel(DecodeParams p, int32_t max_work, PrepParams pp) {
    if (blockIdx.x == 0) {
        plan_body(p, max_work);
        return;
    }
    pdl_wait();
    pdl_trigger();
    const int bi = blockIdx.x - 1;
    if (bi < pp.copy_blocks) {
        copy_token<T>(pp.a, bi * (blockDim.x >> 5) + (threadIdx.x >> 5));
        return;
    }
    const int nsb = gridDim.x - 1 - pp.copy_blocks;
    for (int i = (bi - pp.copy_blocks) * blockDim.x + threadIdx.x; i < pp.r_n; i += nsb * blockDim.x) {
        const float v = pp.R[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        pp.Rhi[i] = hi;
        pp.Rlo[i] = __float2bfloat16_rn(v - __bfloat162float(hi));
    }
}

// The extra per-token key (index_dim elements) into elements [r + d_R, E) of each
// token's row: one warp per token, 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256) append_index_kernel(AppendParams p) {
    pdl_trigger();
    pdl_wait();
    const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= p.num_new) return;
    long long row = 0;
    if (lane == 0) row = locate_slot(p, n);
    row = __shfl_sync(0xffffffffu, row, 0);
    if (row < 0) return;
    constexpr int V = 16 / sizeof(T);
    const int ix = p.s.ix;
    uint4 *dst = (uint4 *)((T *)p.latent + (size_t)row * p.s.E() + p.s.D());
    const uint4 *src = (const uint4 *)((const T *)p.index_key + (size_t)n * ix);
    for (int v = lane; v < ix / V; v += 32) dst[v] = src[v];
}

constexpr int kAT = 16;   // tokens per INT2 append CTA

// One CTA: kAT tokens x one block of output columns (a whole number of groups, at
// most 128), 128 threads. Thread (token quad tq, column quad cq) runs the 16 fp32 fmaf
// chains of tokens 4 tq .. 4 tq + 3 x columns 4 cq .. 4 cq + 3, each k ascending from
// +0 (the encoding definition's order), reading R as 16-byte rows of its four columns
// and the inputs as 16-byte runs of four k, with R staged through shared memory 32 rows
// at a time; then one thread per (token, group) clips, ranges, rounds scale/zero to
// fp16 and packs the codes.
constexpr int kAKC = 32;  // R rows staged per step
constexpr int kAThreads = 128;
template <int COLS>   // COLS: columns per CTA (128, 96 or 64; 0: read `cols`)
__global__ void __launch_bounds__(kAThreads) append_int2_kernel(AppendParams p, int cols_rt) {
    extern __shared__ float sa[];
    const int cols = COLS ? COLS : cols_rt;
    const int r = p.s.r, dR = p.s.dR, gs = p.s.gs;
    const int RD = p.s.RD();          // rotated dims: r, or r + d_R (INT2_JOINT: [c ; k_R])
    const int RDp = (RD + 3) & ~3;    // row stride of the staged inputs (float4 reads)
    const int ng = RD / gs;
    const bool rope_codes = p.s.kind == MLA_KV_INT2_ROT_QR;   // the rope key as unrotated INT2 groups
    const int QD = p.s.QD(), ng_all = QD / gs;
    const int j0 = blockIdx.y * cols;                          // first output column of this CTA
    const int ncol = min(cols, RD - j0);
    float *sc = sa;                   // [kAT][RDp] rotation input (fp32)
    float *sR = sc + kAT * RDp;       // [2][kAKC][cols] rows of R, this CTA's columns
    const int ys = cols + 1;          // row stride of sy: a (token, group) job per lane reads
                                      // 16 tokens' rows on 16 different banks
    float *sy = sR + 2 * kAKC * cols; // [kAT][ys] rotated
    float *sr = sy + kAT * ys;        // INT2_ROT_QR: [kAT][d_R] rope key (fp32)
    __shared__ long long s_row[kAT];
    const int n0 = blockIdx.x * kAT;
    const int tid = threadIdx.x;
    if (tid < kAT) s_row[tid] = (n0 + tid < p.num_new) ? locate_slot(p, n0 + tid) : -1;
    const __nv_bfloat16 *c = (const __nv_bfloat16 *)p.c_kv;
    const __nv_bfloat16 *kr = (const __nv_bfloat16 *)p.k_rope;
    for (int t = 0; t < kAT; ++t)
        for (int k = tid; k < RDp; k += blockDim.x) {
            float v = 0.f;
            if (n0 + t < p.num_new && k < RD)
                v = k < r ? __bfloat162float(c[(size_t)(n0 + t) * r + k]) : __bfloat162float(kr[(size_t)(n0 + t) * dR + k - r]);
            sc[t * RDp + k] = v;
        }
    if (rope_codes && blockIdx.y == 0)
        for (int idx = tid; idx < kAT * dR; idx += blockDim.x) {
            int t = idx / dR, d = idx % dR;
            sr[idx] = (n0 + t < p.num_new) ? __bfloat162float(kr[(size_t)(n0 + t) * dR + d]) : 0.f;
        }
    static_assert(kAT == 16 && kAThreads == 128, "four token quads x 32 column quads");
    const int cq = tid & 31, tq = tid >> 5;                   // column quad, token quad
    const bool act = 4 * cq < ncol;                           // ncol is a multiple of 4
    float acc[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) acc[t][c4] = 0.f;
    const float *scb = sc + (4 * tq) * RDp;
    // R chunks of kAKC rows, double-buffered: chunk c + 1 is read from global memory
    // into registers while chunk c is used, then stored into the other buffer
    constexpr int kPer = kAKC * 128 / kAThreads;              // chunk elements per thread (cols <= 128)
    const int nchunks = (RD + kAKC - 1) / kAKC;
    float pre[kPer];
    auto load_chunk = [&](int k0) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int idx = tid + e * kAThreads, kk = idx / cols, cc = idx % cols;
            pre[e] = (idx < kAKC * cols && k0 + kk < RD && cc < ncol) ? __ldg(p.R + (size_t)(k0 + kk) * RD + j0 + cc) : 0.f;
        }
    };
    auto store_chunk = [&](float *dst) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int idx = tid + e * kAThreads;
            if (idx < kAKC * cols) dst[idx] = pre[e];
        }
    };
    load_chunk(0);
    store_chunk(sR);
    for (int ch = 0; ch < nchunks; ++ch) {
        __syncthreads();              // chunk ch stored (and sc ready on the first pass)
        if (ch + 1 < nchunks) load_chunk((ch + 1) * kAKC);
        const float *sRc = sR + (ch & 1) * kAKC * cols;
        const int k0 = ch * kAKC;
        if (act) {
            const int kn = min(kAKC, RD - k0);      // a multiple of 4 (RD is)
#pragma unroll 2
            for (int kk = 0; kk < kn; kk += 4) {
                float4 rr4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) rr4[u] = *(const float4 *)(sRc + (kk + u) * cols + 4 * cq);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float4 x = *(const float4 *)(scb + t * RDp + k0 + kk);
                    // k ascending within each column's chain: the definition's order
                    acc[t][0] = __fmaf_rn(x.x, rr4[0].x, acc[t][0]);
                    acc[t][1] = __fmaf_rn(x.x, rr4[0].y, acc[t][1]);
                    acc[t][2] = __fmaf_rn(x.x, rr4[0].z, acc[t][2]);
                    acc[t][3] = __fmaf_rn(x.x, rr4[0].w, acc[t][3]);
                    acc[t][0] = __fmaf_rn(x.y, rr4[1].x, acc[t][0]);
                    acc[t][1] = __fmaf_rn(x.y, rr4[1].y, acc[t][1]);
                    acc[t][2] = __fmaf_rn(x.y, rr4[1].z, acc[t][2]);
                    acc[t][3] = __fmaf_rn(x.y, rr4[1].w, acc[t][3]);
                    acc[t][0] = __fmaf_rn(x.z, rr4[2].x, acc[t][0]);
                    acc[t][1] = __fmaf_rn(x.z, rr4[2].y, acc[t][1]);
                    acc[t][2] = __fmaf_rn(x.z, rr4[2].z, acc[t][2]);
                    acc[t][3] = __fmaf_rn(x.z, rr4[2].w, acc[t][3]);
                    acc[t][0] = __fmaf_rn(x.w, rr4[3].x, acc[t][0]);
                    acc[t][1] = __fmaf_rn(x.w, rr4[3].y, acc[t][1]);
                    acc[t][2] = __fmaf_rn(x.w, rr4[3].z, acc[t][2]);
                    acc[t][3] = __fmaf_rn(x.w, rr4[3].w, acc[t][3]);
                }
            }
        }
        if (ch + 1 < nchunks) store_chunk(sR + ((ch + 1) & 1) * kAKC * cols);
    }
    if (act)
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) sy[(4 * tq + t) * ys + 4 * cq + c4] = acc[t][c4];
    __syncthreads();
    // this CTA's groups of the rotated row; INT2_ROT_QR: the rope key's groups in the
    // first column block
    const int g0 = j0 / gs, gn = ncol / gs;
    const int extra = (rope_codes && blockIdx.y == 0) ? ng_all - ng : 0;
    for (int job = tid; job < kAT * (gn + extra); job += blockDim.x) {
        const int t = job % kAT, gl = job / kAT;            // lanes: consecutive tokens
        const long long row = s_row[t];
        if (row < 0) continue;
        const int g = gl < gn ? g0 + gl : ng + (gl - gn);
        const float thr = p.clip[g];
        const float *y = gl < gn ? sy + t * ys + gl * gs : sr + t * dR + (g - ng) * gs;
        float lo = CUDART_INF_F, hi = -CUDART_INF_F;
        for (int j = 0; j < gs; ++j) {
            float v = fminf(fmaxf(y[j], -thr), thr);
            lo = fminf(lo, v);
            hi = fmaxf(hi, v);
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
        const __half z16 = __float2half_rn(lo);
        const float s = __half2float(s16), z = __half2float(z16);
        uint8_t *dst = p.codes + (size_t)row * (QD / 4) + g * (gs / 4);
        for (int j4 = 0; j4 < gs / 4; ++j4) {
            unsigned byte = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = fminf(fmaxf(y[4 * j4 + e], -thr), thr);
                int code = 0;
                if (s != 0.f) {
                    float qv = rintf(__fdiv_rn(__fsub_rn(v, z), s));
                    code = qv < 0.f ? 0 : (qv > 3.f ? 3 : (int)qv);
                }
                byte |= (unsigned)code << (2 * e);
            }
            dst[j4] = (uint8_t)byte;
        }
        __half *szp = p.scale_zero + ((size_t)row * ng_all + g) * 2;
        szp[0] = s16;
        szp[1] = z16;
    }
    if (p.s.kind == MLA_KV_INT2_ROT && blockIdx.y == 0)   // the rope key kept in bf16
        for (int idx = tid; idx < kAT * dR; idx += blockDim.x) {
            const int t = idx / dR, d = idx % dR;
            const long long row = s_row[t];
            if (row >= 0) p.rope[(size_t)row * dR + d] = kr[(size_t)(n0 + t) * dR + d];
        }
}

cudaError_t launch_append_index(const AppendParams &p, cudaStream_t st) {
    if (p.num_new == 0) return cudaSuccess;
    if (p.s.kind == MLA_KV_BF16)
        return launch_pdl(append_index_kernel<__nv_bfloat16>, dim3((p.num_new + 7) / 8), dim3(256), 0, st, p);
    return launch_pdl(append_index_kernel<float>, dim3((p.num_new + 7) / 8), dim3(256), 0, st, p);
}

cudaError_t launch_plan_prep(const DecodeParams &p, int32_t max_work, const AppendParams *a, const float *R,
                             __nv_bfloat16 *Rsplit, int32_t r_n, cudaStream_t st) {
    const int threads = p.B >= 1024 ? 1024 : ((p.B + 31) / 32) * 32;
    int nt = threads > 0 ? threads : 32;
    if (R && nt < 128) nt = 128;                 // the split blocks: eight elements a thread or so
    PrepParams pp;
    memset(&pp, 0, sizeof pp);
    if (a) pp.a = *a;
    const int warps = nt / 32;
    pp.copy_blocks = a ? (a->num_new + warps - 1) / warps : 0;
    int split_blocks = 0;
    if (R) {
        pp.R = R;
        pp.Rhi = Rsplit;
        pp.Rlo = Rsplit + r_n;
        pp.r_n = r_n;
        split_blocks = (r_n + nt * 8 - 1) / (nt * 8);
    }
    const dim3 grid(1 + pp.copy_blocks + split_blocks);
    auto kern = (a && a->s.kind == MLA_KV_FP32) ? plan_prep_kernel<float> : plan_prep_kernel<__nv_bfloat16>;
    return launch_pdl(kern, grid, dim3(nt), (size_t)nt * 28, st, p, max_work, pp);
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t st) {
    if (p.num_new == 0) return cudaSuccess;
    if (p.s.kind == MLA_KV_BF16) {
        return launch_pdl(append_copy_kernel<__nv_bfloat16>, dim3((p.num_new + 7) / 8), dim3(256), 0, st, p);
    } else if (p.s.kind == MLA_KV_FP32) {
        return launch_pdl(append_copy_kernel<float>, dim3((p.num_new + 7) / 8), dim3(256), 0, st, p);
    } else {
        // column blocks of whole groups, at most 128 columns (group_size <= 128): 128,
        // 96 or 64 where that splits the rotated row into whole blocks (compiled), else
        // the largest multiple of the group size up to 128
        const int RD = p.s.RD(), gs = p.s.gs;
        int cols = (128 / gs) * gs;
        for (int c : {128, 96, 64})
            if (c % gs == 0 && RD % c == 0) {
                cols = c;
                break;
            }
        const int RDp = (RD + 3) & ~3;
        const size_t smem = sizeof(float) * ((size_t)kAT * RDp + (size_t)2 * kAKC * cols + (size_t)kAT * (cols + 1) +
                                             (p.s.kind == MLA_KV_INT2_ROT_QR ? (size_t)kAT * p.s.dR : 0));
        dim3 grid((p.num_new + kAT - 1) / kAT, (p.s.RD() + cols - 1) / cols);
        if (cols == 128) {
            cudaFuncSetAttribute(append_int2_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            append_int2_kernel<128><<<grid, kAThreads, smem, st>>>(p, cols);
        } else if (cols == 96) {
            cudaFuncSetAttribute(append_int2_kernel<96>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            append_int2_kernel<96><<<grid, kAThreads, smem, st>>>(p, cols);
        } else if (cols == 64) {
            cudaFuncSetAttribute(append_int2_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            append_int2_kernel<64><<<grid, kAThreads, smem, st>>>(p, cols);
        } else {
            cudaFuncSetAttribute(append_int2_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            append_int2_kernel<0><<<grid, kAThreads, smem, st>>>(p, cols);
        }
    }
    return cudaGetLastError();
}

}  // namespace mla

namespace mla {
// ============================================================================
// Output rotation folded into the up-projection: Wf[h] = R^T . W_UV[h] ([r, r]^T x
// [r, d_v]), fp32 accumulation over k ascending, rounded to bf16. One-time per
// layer. A CTA computes a 64 x 64 tile of one head's output, staging 32-row slabs
// of R and W_UV in shared memory; thread (ty, tx) owns a 4 x 4 block.
// ============================================================================
__global__ void __launch_bounds__(256) fold_rotation_kernel(const float *R, const __nv_bfloat16 *W, __nv_bfloat16 *Wf,
                                                            int r, int dv) {
    __shared__ float sR[32][64 + 1];   // R[k0 + kk][i0 + ii]
    __shared__ float sW[32][64 + 1];   // W[h][k0 + kk][j0 + jj]
    const int h = blockIdx.z, i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const __nv_bfloat16 *Wh = W + (size_t)h * r * dv;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < r; k0 += 32) {
        for (int e = threadIdx.x; e < 32 * 64; e += 256) {
            const int kk = e >> 6, c = e & 63;
            const int k = k0 + kk;
            sR[kk][c] = (k < r && i0 + c < r) ? R[(size_t)k * r + i0 + c] : 0.f;
            sW[kk][c] = (k < r && j0 + c < dv) ? __bfloat162float(Wh[(size_t)k * dv + j0 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < 32; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = sR[kk][4 * ty + u];
                b[u] = sW[kk][4 * tx + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = i0 + 4 * ty + u;
        if (i >= r) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = j0 + 4 * tx + v;
            if (j < dv) Wf[((size_t)h * r + i) * dv + j] = __float2bfloat16_rn(acc[u][v]);
        }
    }
}

cudaError_t launch_fold_rotation(const ShapeArgs &s, const float *R, const void *W_UV, void *W_folded, cudaStream_t st) {
    dim3 grid((s.dv + 63) / 64, (s.r + 63) / 64, s.H);
    fold_rotation_kernel<<<grid, 256, 0, st>>>(R, (const __nv_bfloat16 *)W_UV, (__nv_bfloat16 *)W_folded, s.r, s.dv);
    return cudaGetLastError();
}
}  // namespace mla
