// C ABI entry points: argument checks, the workspace layout, implementation
// choice and the launch sequence of append, decode and verify.
#include "mla_internal.cuh"

#include <string.h>

namespace mla {

static int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// ---- benchmarking diagnostics (see mla_profile_enable) ----------------------
struct Profile {
    bool on = false;
    bool events = true;       // record the event pairs (mode 1) or only count launches (mode 2)
    int32_t kernels = 0;
    int32_t used = 0;
    static constexpr int kMax = 1 << 14;
    cudaEvent_t start[kMax];
    cudaEvent_t stop[kMax];
    int32_t created = 0;
};
static Profile g_prof;

// Records the start event of the next pair; returns the pair index or -1.
static int prof_begin(cudaStream_t st) {
    if (!g_prof.on || !g_prof.events || g_prof.used >= Profile::kMax) return -1;
    const int i = g_prof.used;
    if (i >= g_prof.created) {
        if (cudaEventCreate(&g_prof.start[i]) != cudaSuccess) return -1;
        if (cudaEventCreate(&g_prof.stop[i]) != cudaSuccess) return -1;
        g_prof.created = i + 1;
    }
    cudaEventRecord(g_prof.start[i], st);
    g_prof.used = i + 1;
    return i;
}
static void prof_end(int i, cudaStream_t st) {
    if (i >= 0) cudaEventRecord(g_prof.stop[i], st);
}
static void prof_kernels(int n) {
    if (g_prof.on) g_prof.kernels += n;
}

// Shape checks shared by every entry point.
static mla_status check_shape(const mla_shape *s) {
    if (!s) return MLA_ERR_INVALID;
    if (s->num_heads < 1 || s->kv_lora_rank < 8 || s->kv_lora_rank % 8 || s->rope_dim < 0 ||
        s->rope_dim % 8 || s->v_head_dim < 1 || s->block_size < 1 || s->num_blocks < 1)
        return MLA_ERR_INVALID;
    if (s->kind != MLA_KV_BF16 && s->kind != MLA_KV_FP32 && !is_int2(s->kind)) return MLA_ERR_INVALID;
    if (s->impl < MLA_IMPL_AUTO || s->impl > MLA_IMPL_TCGEN05 || s->num_splits_hint < 0)
        return MLA_ERR_INVALID;
    if (s->index_dim < 0 || s->index_dim % 8 || s->index_dim > 1024) return MLA_ERR_INVALID;
    if (is_int2(s->kind) && s->index_dim != 0) return MLA_ERR_INVALID;
    if (s->flags & ~(int32_t)(MLA_FLAG_WUV_FOLDED | MLA_FLAG_Q_ROTATED)) return MLA_ERR_INVALID;
    // the joint kind's folded up-projection would be [H, r + d_R, d_v]: not offered
    if ((s->flags & (MLA_FLAG_WUV_FOLDED | MLA_FLAG_Q_ROTATED)) && (!is_int2(s->kind) || s->kind == MLA_KV_INT2_JOINT))
        return MLA_ERR_INVALID;
    if (is_int2(s->kind)) {
        if (s->group_size < 4 || s->group_size > 128 || s->group_size % 4 || s->kv_lora_rank % s->group_size)
            return MLA_ERR_INVALID;
        if (s->rope_dim < 8) return MLA_ERR_INVALID;
        if ((s->kind == MLA_KV_INT2_ROT_QR || s->kind == MLA_KV_INT2_JOINT) && s->rope_dim % s->group_size)
            return MLA_ERR_INVALID;
    }
    // generic kernel limits (shared-memory tiles sized from r and d_R)
    if (s->kv_lora_rank > 1024 || s->rope_dim > 128) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

static ShapeArgs shape_args(const mla_shape *s) {
    ShapeArgs a;
    a.H = s->num_heads;
    a.r = s->kv_lora_rank;
    a.dR = s->rope_dim;
    a.dv = s->v_head_dim;
    a.bs = s->block_size;
    a.num_blocks = s->num_blocks;
    a.gs = s->group_size;
    a.kind = s->kind;
    a.ix = is_int2(s->kind) ? 0 : s->index_dim;
    return a;
}

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

int32_t resolve_impl(const mla_shape *s, int32_t q_len) {
    (void)q_len;
    const bool tc_ok = tc_shape_supported(shape_args(s));
    if (s->impl == MLA_IMPL_TCGEN05) return tc_ok ? (int32_t)MLA_IMPL_TCGEN05 : (int32_t)MLA_ERR_UNSUPPORTED;
    if (s->impl == MLA_IMPL_SIMT) return MLA_IMPL_SIMT;
    return tc_ok ? MLA_IMPL_TCGEN05 : MLA_IMPL_SIMT;
}

// Units the planner charges per sequence start on the tensor-core path (a work item's
// query load and epilogue cost about as much as two to three 64-token tiles, or one
// to two 128-token steps of the bf16 decode that scores two blocks per MMA).
constexpr int kItemCostTc = 3;
constexpr int kItemCostWide = 2;
// mla_append_decode: new tokens up to this count are copied by the planner's launch
constexpr int32_t kFusedAppendMax = 4096;

static WsLayout ws_layout(const mla_shape *s, int32_t B, int32_t q_len, int32_t impl) {
    WsLayout w;
    memset(&w, 0, sizeof w);
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    int target;
    if (impl == MLA_IMPL_TCGEN05) {
        // one wave of persistent CTAs: 2 per stream per 128-row tile
        const int row_tiles = (q_len * s->num_heads + 127) / 128;
        target = sms / (2 * row_tiles);
        if (target < 1) target = 1;
        if (s->num_splits_hint > 0 && s->num_splits_hint < target) target = s->num_splits_hint;
    } else {
        target = s->num_splits_hint > 0 ? s->num_splits_hint : sms;
    }
    w.target = target;
    w.max_work = target + B;
    const size_t rows = (size_t)q_len * s->num_heads;
    size_t off = 0;
    w.status = off;        off = up256(off + 2 * sizeof(int32_t));
    w.work = off;          off = up256(off + sizeof(WorkItem) * (size_t)w.max_work);
    w.split_start = off;   off = up256(off + sizeof(int32_t) * ((size_t)B + 1));
    w.stream_start = off;  off = up256(off + sizeof(int32_t) * ((size_t)target + 1));
    w.part_o = off;        off = up256(off + sizeof(float) * (size_t)w.max_work * rows * shape_args(s).OD());
    w.part_lse = off;      off = up256(off + sizeof(float) * (size_t)w.max_work * rows);
    w.q_prep = off;
    if (is_int2(s->kind)) {
        const size_t nrow = (size_t)B * rows;
        off = up256(off + sizeof(float) * nrow * (s->kv_lora_rank + s->rope_dim));
        w.o_rot = off;  off = up256(off + sizeof(float) * nrow * s->kv_lora_rank);
        w.o_lat = off;  off = up256(off + sizeof(float) * nrow * s->kv_lora_rank);
        w.lse2 = off;   off = up256(off + sizeof(float) * nrow);
        w.ident = off;  off = up256(off + sizeof(int32_t) * ((size_t)B + 1));
        w.r16 = off;    off = up256(off + sizeof(__half) * (size_t)s->kv_lora_rank * s->kv_lora_rank);
        w.rsplit = off; off = up256(off + 2 * sizeof(__nv_bfloat16) * (size_t)s->kv_lora_rank * s->kv_lora_rank);
    }
    w.total = off;
    return w;
}

// `fuse`: the step's new tokens, appended before the attention (mla_append_decode);
// nullptr for a plain decode or verify. Its arguments are checked by the caller.
static mla_status run_attention(const mla_shape *s, const mla_cache *cache, const int32_t *block_table,
                                int32_t max_blocks, const int32_t *seq_lens, int32_t B, int32_t q_len,
                                const void *q, const void *W_UV, const float *R, float scale, void *out,
                                float *lse, void *workspace, size_t ws_bytes, void *stream,
                                const AppendParams *fuse = nullptr) {
    mla_status st = check_shape(s);
    if (st != MLA_OK) return st;
    if (!cache || !block_table || !seq_lens || !q || !W_UV || !out || !lse || !workspace) return MLA_ERR_INVALID;
    if (B < 1 || q_len < 1 || max_blocks < 1) return MLA_ERR_INVALID;
    if (!(scale == scale)) return MLA_ERR_INVALID;
    const bool int2 = is_int2(s->kind);
    const bool rope_bf16 = s->kind == MLA_KV_INT2_ROT;      // INT2_ROT_QR holds the rope key as codes
    if (int2) {
        // R is read for the query (unless it comes rotated) and for the output (unless
        // W_UV comes folded)
        const bool r_unused = (s->flags & MLA_FLAG_WUV_FOLDED) && (s->flags & MLA_FLAG_Q_ROTATED);
        if (!cache->codes || !cache->scale_zero || (rope_bf16 && !cache->rope) || (!R && !r_unused))
            return MLA_ERR_INVALID;
        if (!aligned16(cache->codes) || !aligned16(cache->scale_zero) || (rope_bf16 && !aligned16(cache->rope)))
            return MLA_ERR_INVALID;
    } else {
        if (!cache->latent || !aligned16(cache->latent)) return MLA_ERR_INVALID;
    }
    if (!aligned16(q) || !aligned16(workspace)) return MLA_ERR_INVALID;
    const int32_t impl = resolve_impl(s, q_len);
    if (impl < 0) return (mla_status)impl;
    const WsLayout w = ws_layout(s, B, q_len, impl);
    if (ws_bytes < w.total) return MLA_ERR_WORKSPACE;
    cudaStream_t stream_ = (cudaStream_t)stream;
    char *ws = (char *)workspace;

    DecodeParams p;
    memset(&p, 0, sizeof p);
    p.s = shape_args(s);
    p.B = B;
    p.q_len = q_len;
    p.max_blocks = max_blocks;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.latent = cache->latent;
    p.codes = (const uint8_t *)cache->codes;
    p.scale_zero = (const __half *)cache->scale_zero;
    p.rope = (const __nv_bfloat16 *)cache->rope;
    p.q = q;
    p.q_rope = q;
    p.q_prep = int2 ? (const float *)(ws + w.q_prep) : nullptr;
    p.scale_log2 = scale * kLog2e;
    p.status = (int32_t *)(ws + w.status);
    p.num_work = (const int32_t *)(ws + w.status + sizeof(int32_t));
    // the bf16 decode that scores two blocks per MMA plans in 128-token steps, so that
    // only a sequence's last work item can end with an unpaired block
    const bool wide = impl == MLA_IMPL_TCGEN05 && s->kind == MLA_KV_BF16;
    p.item_cost = impl == MLA_IMPL_TCGEN05 ? (wide ? kItemCostWide : kItemCostTc) : 0;
    p.plan_tile = wide ? 128 : 64;
    p.work = (const WorkItem *)(ws + w.work);
    p.split_start = (const int32_t *)(ws + w.split_start);
    p.stream_start = (const int32_t *)(ws + w.stream_start);
    p.streams = w.target;
    p.part_o = (float *)(ws + w.part_o);
    p.part_lse = (float *)(ws + w.part_lse);

    const bool tc = impl == MLA_IMPL_TCGEN05;
    // Work that needs nothing from the planner rides on its launch: a decode step's few
    // new tokens (bf16 / fp32 cache; otherwise the append runs as its own kernel first)
    // and the split of R for the tensor-core query rotation.
    int launches = 0;
    const bool copy_fused = fuse && !int2 && fuse->num_new <= kFusedAppendMax;
    const bool split_fused = int2 && tc && !(s->flags & MLA_FLAG_Q_ROTATED);
    if (fuse && !copy_fused) {
        if (launch_append(*fuse, stream_) != cudaSuccess) return MLA_ERR_CUDA;
        ++launches;
    }
    if (copy_fused || split_fused) {
        if (launch_plan_prep(p, w.max_work, copy_fused ? fuse : nullptr, split_fused ? R : nullptr,
                             (__nv_bfloat16 *)(ws + w.rsplit), s->kv_lora_rank * s->kv_lora_rank,
                             stream_) != cudaSuccess)
            return MLA_ERR_CUDA;
    } else if (launch_plan(p, w.max_work, stream_) != cudaSuccess) {
        return MLA_ERR_CUDA;
    }
    if (int2) {
        // the rotated query: fp32 for the CUDA-core kernel; fp16 (the MMA operand type
        // of this cache kind) from the tensor-core GEMM for the tensor-core kernel,
        // which then reads it in place of q
        if (s->flags & MLA_FLAG_Q_ROTATED) {
            // already rotated: only widened to the operand type (fp16 for the tensor
            // cores, fp32 for the CUDA-core kernel)
            if (launch_convert_query(q, ws + w.q_prep, (size_t)B * q_len * s->num_heads * p.s.D(), tc, stream_) !=
                cudaSuccess)
                return MLA_ERR_CUDA;
            if (tc) p.q = ws + w.q_prep;
        } else if (tc) {
            if (launch_rot_query(R, (__nv_bfloat16 *)(ws + w.rsplit), q, ws + w.q_prep, B * q_len * s->num_heads,
                                 s->kv_lora_rank + s->rope_dim, p.status, stream_, split_fused) != cudaSuccess)
                return MLA_ERR_CUDA;
            p.q = ws + w.q_prep;
        } else if (launch_qprep(p, R, ws + w.q_prep, false, stream_) != cudaSuccess) {
            return MLA_ERR_CUDA;
        }
    }
    const int ev = prof_begin(stream_);
    const cudaError_t de = impl == MLA_IMPL_TCGEN05 ? launch_decode_tc(p, w.max_work, stream_)
                                                    : launch_decode_simt(p, w.max_work, stream_);
    if (de != cudaSuccess) return MLA_ERR_CUDA;
    prof_end(ev, stream_);

    CombineParams c;
    memset(&c, 0, sizeof c);
    c.s = p.s;
    c.B = B;
    c.q_len = q_len;
    c.split_start = p.split_start;
    c.part_bf16 = impl == MLA_IMPL_TCGEN05;   // the tensor-core decode writes bf16 partials
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.R = int2 ? R : nullptr;
    c.W_UV = W_UV;
    c.out = out;
    c.lse = lse;
    const bool comb_tc = tc && combine_tc_supported(p.s);
    // the tensor-core decode kernels release the combine only after their own wait for
    // the planner, whose split ranges the combine may then read before its wait
    c.ranges_early = tc ? 1 : 0;
    const bool folded = int2 && (s->flags & MLA_FLAG_WUV_FOLDED);
    if (folded) c.R = nullptr;                 // W_UV already carries R^T
    if (int2 && comb_tc && !folded) {
        // merge splits, rotate back on the tensor cores (o_lat = o_rot . R^T), then the
        // W_UV up-projection reads the merged rows as one-split partials
        float *o_rot = (float *)(ws + w.o_rot), *o_lat = (float *)(ws + w.o_lat), *lse2 = (float *)(ws + w.lse2);
        int32_t *ident = (int32_t *)(ws + w.ident);
        if (launch_rot_output(c, (__half *)(ws + w.r16), o_rot, o_lat, lse2, ident, p.status, stream_) !=
            cudaSuccess)
            return MLA_ERR_CUDA;
        c.split_start = ident;
        c.ranges_early = 0;                    // written by the merge, two kernels back
        c.part_bf16 = 0;                       // o_lat is fp32
        c.part_o = o_lat;
        c.part_lse = lse2;
        c.R = nullptr;
        if (launch_combine_tc(c, stream_) != cudaSuccess) return MLA_ERR_CUDA;
        launches += 3;              // merge, R to fp16, o . R^T
    } else {
        if ((comb_tc ? launch_combine_tc(c, stream_) : launch_combine(c, stream_)) != cudaSuccess) return MLA_ERR_CUDA;
    }
    // plan, decode, combine; INT2 adds the query preparation: the tensor-core rotation
    // (R split + GEMM), the CUDA-core one, or the conversion of a query given rotated
    launches += 3;
    if (int2) launches += 1;    // the query rotation (R split by the planner's launch) or conversion
    prof_kernels(launches);
    return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_workspace_bytes(const mla_shape *shape, int32_t B, int32_t q_len) {
    if (check_shape(shape) != MLA_OK || B < 1 || q_len < 1) return 0;
    const int32_t impl = resolve_impl(shape, q_len);
    if (impl < 0) return 0;
    return ws_layout(shape, B, q_len, impl).total;
}

// Checks of mla_latent_append's arguments (num_new > 0) and its kernel parameters.
static mla_status append_params(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                                int32_t max_blocks_per_seq, int32_t B, const int32_t *start_pos,
                                const int32_t *cu_new, int32_t num_new, const void *c_kv, const void *k_rope,
                                const float *R, const float *clip, int32_t *status, AppendParams &p) {
    if (!c_kv || !k_rope || !aligned16(c_kv) || !aligned16(k_rope)) return MLA_ERR_INVALID;
    const bool int2 = is_int2(shape->kind);
    if (int2) {
        if (!cache->codes || !cache->scale_zero || (shape->kind == MLA_KV_INT2_ROT && !cache->rope) || !R || !clip)
            return MLA_ERR_INVALID;
    } else {
        if (!cache->latent || !aligned16(cache->latent)) return MLA_ERR_INVALID;
    }
    memset(&p, 0, sizeof p);
    p.s = shape_args(shape);
    p.B = B;
    p.max_blocks = max_blocks_per_seq;
    p.num_new = num_new;
    p.block_table = block_table;
    p.start_pos = start_pos;
    p.cu_new = cu_new;
    p.c_kv = c_kv;
    p.k_rope = k_rope;
    p.R = R;
    p.clip = clip;
    p.latent = cache->latent;
    p.codes = (uint8_t *)cache->codes;
    p.scale_zero = (__half *)cache->scale_zero;
    p.rope = (__nv_bfloat16 *)cache->rope;
    p.status = status;
    return MLA_OK;
}

mla_status mla_latent_append(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                             int32_t max_blocks_per_seq, int32_t B, const int32_t *start_pos,
                             const int32_t *cu_new, int32_t num_new, const void *c_kv, const void *k_rope,
                             const float *R, const float *clip, int32_t *status, void *stream) {
    mla_status st = check_shape(shape);
    if (st != MLA_OK) return st;
    if (!cache || !block_table || !start_pos || !cu_new || B < 1 || max_blocks_per_seq < 1 || num_new < 0)
        return MLA_ERR_INVALID;
    if (num_new == 0) return MLA_OK;
    AppendParams p;
    st = append_params(shape, cache, block_table, max_blocks_per_seq, B, start_pos, cu_new, num_new, c_kv, k_rope,
                       R, clip, status, p);
    if (st != MLA_OK) return st;
    if (launch_append(p, (cudaStream_t)stream) != cudaSuccess) return MLA_ERR_CUDA;
    prof_kernels(1);
    return MLA_OK;
}

mla_status mla_append_decode(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                             int32_t max_blocks_per_seq, int32_t B, const int32_t *start_pos,
                             const int32_t *cu_new, int32_t num_new, const void *c_kv, const void *k_rope,
                             const float *clip, int32_t *append_status, const int32_t *seq_lens, const void *q,
                             const void *W_UV, const float *R, float scale, void *out, float *lse, void *workspace,
                             size_t workspace_bytes, void *stream) {
    mla_status st = check_shape(shape);
    if (st != MLA_OK) return st;
    if (!cache || !block_table || !start_pos || !cu_new || B < 1 || max_blocks_per_seq < 1 || num_new < 0)
        return MLA_ERR_INVALID;
    AppendParams a;
    if (num_new > 0) {
        st = append_params(shape, cache, block_table, max_blocks_per_seq, B, start_pos, cu_new, num_new, c_kv,
                           k_rope, R, clip, append_status, a);
        if (st != MLA_OK) return st;
    }
    return run_attention(shape, cache, block_table, max_blocks_per_seq, seq_lens, B, 1, q, W_UV, R, scale, out, lse,
                         workspace, workspace_bytes, stream, num_new > 0 ? &a : nullptr);
}

mla_status mla_latent_append_index(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, int32_t B, const int32_t *start_pos,
                                   const int32_t *cu_new, int32_t num_new, const void *index_key,
                                   int32_t *status, void *stream) {
    mla_status st = check_shape(shape);
    if (st != MLA_OK) return st;
    if (is_int2(shape->kind) || shape->index_dim == 0) return MLA_ERR_INVALID;
    if (!cache || !block_table || !start_pos || !cu_new || B < 1 || max_blocks_per_seq < 1 || num_new < 0)
        return MLA_ERR_INVALID;
    if (num_new == 0) return MLA_OK;
    if (!index_key || !aligned16(index_key) || !cache->latent || !aligned16(cache->latent)) return MLA_ERR_INVALID;
    AppendParams p;
    memset(&p, 0, sizeof p);
    p.s = shape_args(shape);
    p.B = B;
    p.max_blocks = max_blocks_per_seq;
    p.num_new = num_new;
    p.block_table = block_table;
    p.start_pos = start_pos;
    p.cu_new = cu_new;
    p.index_key = index_key;
    p.latent = cache->latent;
    p.status = status;
    if (launch_append_index(p, (cudaStream_t)stream) != cudaSuccess) return MLA_ERR_CUDA;
    prof_kernels(1);
    return MLA_OK;
}

mla_status mla_decode(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, const void *q,
                      const void *W_UV, const float *R, float scale, void *out, float *lse, void *workspace,
                      size_t workspace_bytes, void *stream) {
    return run_attention(shape, cache, block_table, max_blocks_per_seq, seq_lens, B, 1, q, W_UV, R, scale, out,
                         lse, workspace, workspace_bytes, stream);
}

mla_status mla_verify(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t q_len,
                      const void *q, const void *W_UV, const float *R, float scale, void *out, float *lse,
                      void *workspace, size_t workspace_bytes, void *stream) {
    return run_attention(shape, cache, block_table, max_blocks_per_seq, seq_lens, B, q_len, q, W_UV, R, scale,
                         out, lse, workspace, workspace_bytes, stream);
}

static mla_status flags_to_status(int32_t f) {
    if (f & FLAG_TIMEOUT) return MLA_ERR_TIMEOUT;
    if (f & (FLAG_BAD_BLOCK | FLAG_BAD_LENGTH)) return MLA_ERR_BOUNDS;
    return MLA_OK;
}

mla_status mla_read_status_word(const int32_t *status, int32_t *raw_flags, void *stream) {
    if (!status) return MLA_ERR_INVALID;
    int32_t f = 0;
    if (cudaMemcpyAsync(&f, status, sizeof f, cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MLA_ERR_CUDA;
    if (raw_flags) *raw_flags = f;
    return flags_to_status(f);
}

mla_status mla_get_status(const void *workspace, int32_t *raw_flags, void *stream) {
    // The flags word sits at offset 0 of every workspace layout.
    return mla_read_status_word((const int32_t *)workspace, raw_flags, stream);
}

const char *mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported shape or implementation";
        case MLA_ERR_BOUNDS: return "block id or sequence length out of range (device flag)";
        case MLA_ERR_WORKSPACE: return "workspace too small";
        case MLA_ERR_CUDA: return "CUDA launch or runtime error";
        case MLA_ERR_TIMEOUT: return "bounded device wait gave up (device flag)";
    }
    return "unknown status";
}

int32_t mla_resolve_impl(const mla_shape *shape, int32_t q_len) {
    mla_status st = check_shape(shape);
    if (st != MLA_OK) return st;
    if (q_len < 1) return MLA_ERR_INVALID;
    return resolve_impl(shape, q_len);
}

mla_status mla_profile_enable(int32_t enable) {
    g_prof.on = enable != 0;
    g_prof.events = enable != 2;
    g_prof.used = 0;
    g_prof.kernels = 0;
    return MLA_OK;
}

mla_status mla_profile_read(double *attention_ms, int32_t *attention_launches, int32_t *kernel_launches) {
    double total = 0.0;
    for (int i = 0; i < g_prof.used; ++i) {
        if (cudaEventSynchronize(g_prof.stop[i]) != cudaSuccess) return MLA_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]) != cudaSuccess) return MLA_ERR_CUDA;
        total += ms;
    }
    if (attention_ms) *attention_ms = total;
    if (attention_launches) *attention_launches = g_prof.used;
    if (kernel_launches) *kernel_launches = g_prof.kernels;
    return MLA_OK;
}

mla_status mla_fold_rotation(const mla_shape *shape, const float *R, const void *W_UV, void *W_folded,
                             void *stream) {
    mla_status st = check_shape(shape);
    if (st != MLA_OK) return st;
    if (!is_int2(shape->kind) || shape->kind == MLA_KV_INT2_JOINT || !R || !W_UV || !W_folded || W_UV == W_folded)
        return MLA_ERR_INVALID;
    if (launch_fold_rotation(shape_args(shape), R, W_UV, W_folded, (cudaStream_t)stream) != cudaSuccess)
        return MLA_ERR_CUDA;
    prof_kernels(1);
    return MLA_OK;
}

int32_t mla_version(void) { return 104; }

}  // extern "C"
