// Internal declarations shared by the library's translation units (not part
// of the ABI). Kernel parameter blocks, the workspace layout and small device
// helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// Device status flags (OR-ed into the status word).
enum : int32_t {
    FLAG_BAD_BLOCK = 1,      // a block id outside [0, num_blocks) or a logical block past the table
    FLAG_BAD_LENGTH = 2,     // a sequence length outside [q_len, max_blocks * block_size]
    FLAG_TIMEOUT = 4,        // a bounded wait gave up
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Work item of the split-KV schedule: tokens [t0, t1) of sequence b, processed
// by work stream `stream`. Its partial result goes to the slot equal to its
// index in the schedule; the items of one sequence have consecutive indices,
// and so do the items of one stream.
struct WorkItem {
    int32_t b, t0, t1, stream;
};

// Byte offsets inside the caller's workspace.
struct WsLayout {
    size_t status;        // int32 flags word, then int32 num_work
    size_t work;          // WorkItem[max_work]
    size_t split_start;   // int32[B + 1]: first slot of each sequence
    size_t stream_start;  // int32[streams + 1]: first item of each stream
    size_t part_o;        // [max_work][q_len * H][r] normalised partial outputs: bf16 from the
                          // tensor-core decode, fp32 from the CUDA-core decode (sized for fp32)
    size_t part_lse;      // fp32 [max_work][q_len * H]     partial log2-sum-exp
    size_t q_prep;        // fp32 [B * q_len * H][r + d_R]  rotated query (INT2 kind)
    size_t o_rot;         // fp32 [B * q_len * H][r]  merged rotated output (INT2, tensor cores)
    size_t o_lat;         // fp32 [B * q_len * H][r]  o_rot . R^T
    size_t lse2;          // fp32 [B * q_len * H]     merged log2-sum-exp
    size_t ident;         // int32 [B + 1]           one slot per sequence
    size_t r16;           // fp16 [r][r]             R as the output rotation's operand (INT2, tensor cores)
    size_t rsplit;        // bf16 [2][r][r]          R as two bf16 halves for the query rotation
    size_t total;
    int32_t max_work;     // upper bound of schedule length (streams + B)
    int32_t target;       // number of work streams
};

struct ShapeArgs {
    int32_t H, r, dR, dv, bs, num_blocks, gs, kind;
    int32_t ix;                  // extra per-token key after the rope key (BF16/FP32 kinds)
    __host__ __device__ int32_t D() const { return r + dR; }        // elements attention reads
    __host__ __device__ int32_t E() const { return r + dR + ix; }   // cache row stride (BF16/FP32)
    // INT2 kinds: dims held as codes per token (the latent; INT2_ROT_QR and INT2_JOINT:
    // + the rope key)
    __host__ __device__ int32_t QD() const { return kind == MLA_KV_INT2_ROT_QR || kind == MLA_KV_INT2_JOINT ? r + dR : r; }
    // INT2 kinds: dims the rotation acts on (R is [RD, RD]): the latent, or for
    // INT2_JOINT the whole row [c ; k_R]
    __host__ __device__ int32_t RD() const { return kind == MLA_KV_INT2_JOINT ? r + dR : r; }
    // dims of the attention's latent-space output (the split partials): r, or for
    // INT2_JOINT all r + d_R rotated dims (rotated back and cut to r in the combine)
    __host__ __device__ int32_t OD() const { return kind == MLA_KV_INT2_JOINT ? r + dR : r; }
};

__host__ __device__ constexpr bool is_int2(int32_t kind) {
    return kind == MLA_KV_INT2_ROT || kind == MLA_KV_INT2_ROT_QR || kind == MLA_KV_INT2_JOINT;
}

// Everything a decode kernel reads.
struct DecodeParams {
    ShapeArgs s;
    int32_t B, q_len, max_blocks;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const void *latent;          // BF16 / FP32 kinds
    const uint8_t *codes;        // INT2
    const __half *scale_zero;    // INT2
    const __nv_bfloat16 *rope;   // INT2
    const void *q;               // caller's absorbed query
    const void *q_rope;          // the caller's bf16 query, whose rope dims the tensor-core
                                 // INT2_ROT decode reads as they are (the query itself)
    const float *q_prep;         // INT2: rotated query (fp32), else nullptr
    float scale_log2;            // scale * log2(e)
    int32_t *status;             // -> flags word
    const int32_t *num_work;
    const WorkItem *work;
    const int32_t *split_start;
    const int32_t *stream_start;
    int32_t streams;
    int32_t item_cost;           // planner: units charged per sequence start (its Q load, epilogue)
    int32_t plan_tile;           // planner: tokens per cost unit; work items start at multiples of it
    float *part_o;
    float *part_lse;
};

struct CombineParams {
    ShapeArgs s;
    int32_t B, q_len;
    int32_t part_bf16;           // part_o holds bf16 values (else fp32)
    const int32_t *split_start;
    const void *part_o;
    const float *part_lse;
    int32_t ranges_early;        // split_start comes from the planner and the kernel before the
                                 // combine released it only after its own dependency wait, so
                                 // the planner's writes may be read before the combine's wait
    const float *R;              // INT2: [r, r], else nullptr
    const void *W_UV;            // [H, r, dv]
    void *out;                   // [B, q_len, H, dv]
    float *lse;                  // [B, q_len, H]
};

struct AppendParams {
    ShapeArgs s;
    int32_t B, max_blocks, num_new;
    const int32_t *block_table;
    const int32_t *start_pos;
    const int32_t *cu_new;
    const void *c_kv;
    const void *k_rope;
    const void *index_key;       // mla_latent_append_index: [num_new, ix]; else nullptr
    const float *R;
    const float *clip;
    void *latent;
    uint8_t *codes;
    __half *scale_zero;
    __nv_bfloat16 *rope;
    int32_t *status;
};

// ---- launchers (defined in mla_simt.cu) ------------------------------------
// Programmatic dependent launch. A kernel launched with launch_pdl may start while
// the previous kernel of the stream is still running; it calls pdl_trigger() on entry
// (so that the next kernel may be scheduled as soon as SMs free up) and pdl_wait()
// before its first access to any buffer that another kernel writes or reads.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_plan(const DecodeParams &p, int32_t max_work, cudaStream_t st);
// The planner plus, in the same launch, the bf16 / fp32 copy of a step's new tokens
// (a; nullptr: none) and the split of R ([r_n] fp32) into bf16 halves at Rsplit and
// Rsplit + r_n (R nullptr: none).
cudaError_t launch_plan_prep(const DecodeParams &p, int32_t max_work, const AppendParams *a, const float *R,
                             __nv_bfloat16 *Rsplit, int32_t r_n, cudaStream_t st);
// q (bf16) -> fp16 (out_f16) or fp32, n elements, for a query that comes rotated.
cudaError_t launch_convert_query(const void *q, void *out, size_t n, bool out_f16, cudaStream_t st);
cudaError_t launch_qprep(const DecodeParams &p, const float *R, void *q_prep, bool out_f16, cudaStream_t st);
cudaError_t launch_decode_simt(const DecodeParams &p, int32_t max_work, cudaStream_t st);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t st);
cudaError_t launch_append(const AppendParams &p, cudaStream_t st);
cudaError_t launch_append_index(const AppendParams &p, cudaStream_t st);
cudaError_t launch_fold_rotation(const ShapeArgs &s, const float *R, const void *W_UV, void *W_folded, cudaStream_t st);
// ---- tensor-core decode (defined in mla_tc.cu) -----------------------------
bool tc_shape_supported(const ShapeArgs &s);
cudaError_t launch_decode_tc(const DecodeParams &p, int32_t max_work, cudaStream_t st);
// ---- bf16 tensor-core decode, two cache blocks per score MMA (mla_wide.cu) ----
cudaError_t launch_decode_wide(const DecodeParams &p, int32_t max_work, cudaStream_t st);
// ---- tensor-core combine + W_UV (defined in mla_combine_tc.cu) --------------
bool combine_tc_supported(const ShapeArgs &s);
cudaError_t launch_combine_tc(const CombineParams &c, cudaStream_t st);
// ---- tensor-core rotations of the rotated-INT2 cache (defined in mla_rot_tc.cu)
bool rot_tc_supported(const ShapeArgs &s);
// launch_rot_query writes Rsplit = [bf16(R) ; bf16(R - bf16(R))] ([2][r][r]) first;
// launch_rot_output writes R16 = fp16(R) ([r][r]) first. Both 16-byte aligned.
cudaError_t launch_rot_query(const float *R, __nv_bfloat16 *Rsplit, const void *q_bf16, void *q_rot_f16, int rows,
                             int D, int32_t *status, cudaStream_t st, bool split_done = false);
cudaError_t launch_rot_output(const CombineParams &c, __half *R16, float *o_rot, float *o_lat, float *lse2,
                              int32_t *ident, int32_t *status, cudaStream_t st);

// ---- small device helpers ---------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Four bf16 values (8 bytes, memory order) widened to fp32.
__device__ __forceinline__ float4 bf16x4_to_float4(uint2 u) {
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ void raise_flag(int32_t *status, int32_t f) {
    if (status) atomicOr(status, f);
}

}  // namespace mla
