/*
 * mla.h - C ABI of the GB300 (sm_103a) MLA latent-cache decode library.
 *
 * Multi-head latent attention decode over a paged, compressed latent KV cache
 * in the DeepSeek "absorb" form. Each cached token holds one shared latent c
 * (kv_lora_rank = r elements) and one shared rope key k_R (qk_rope_head_dim =
 * d_R elements); the query arrives already absorbed through W_UK, scores and
 * softmax run against [c ; k_R], and the latent-space output is up-projected
 * per head through W_UV.
 *   Source: "GLM-5.2 speculative drafting: native MTP head beats GLM-4-9B, +
 *   opt-in MLA-latent KV cache" (leyten/shard PR #5), TL;DR item 2; per-token
 *   footprint r + d_R from "hf: size GLM-5.3-Flash's KV cache from its latent
 *   layers only" (coder/llm-helper PR #64), PR description.
 * An opt-in cache kind stores the latent rotated by a per-layer orthogonal
 * covariance eigenbasis R and quantised to grouped INT2 (rope key kept bf16).
 *   Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
 *   maintainer reply, "How the rotation adapts to the latent".
 * Two variants also quantise the rope key, the two rope/nope designs the same
 * thread names as benchmarked, without details (a later reply on GLM-5.2
 * support): MLA_KV_INT2_ROT_QR keeps the rope key unrotated as further INT2
 * groups; MLA_KV_INT2_JOINT rotates the latent and the rope key together by one
 * eigenbasis of the whole row and quantises the result.
 *
 * Definitions (per sequence b, query row i, head h, cached token t):
 *   s = scale * (q[b,i,h,:] . [c_t ; kR_t])          (rotated kind: q_lat . R)
 *   visible t: 0 <= t <= L_b - q_len + i               (causal draft window)
 *   lse[b,i,h] = ln sum_visible exp(s)
 *   olat = sum_t softmax(s)_t c_t                      (rotated kind: . R^T)
 *   out[b,i,h,:] = olat . W_UV[h]                      ([r] x [r, d_v])
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers on the current CUDA device unless the
 *     argument says "host". The caller owns every buffer; no call allocates
 *     device memory, and none synchronises (mla_get_status is the one call
 *     that waits, on the given stream). The one piece of device memory the
 *     library holds itself is the fixed 32 MiB scratch array of
 *     mla_decode_noalloc, a static device variable that exists on every GPU
 *     where the library's module is loaded, for as long as it stays loaded.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *     stream. Work is enqueued on it and the call returns immediately.
 *   - Row-major, densely packed layouts as stated per argument. Device buffers
 *     must be 16-byte aligned.
 *   - Host-side argument errors return before anything is launched. Device-side
 *     problems (a block id outside [0, num_blocks), a sequence length outside
 *     [q_len, max_blocks_per_seq * block_size]) never trap: the kernel records
 *     a flag, skips the bad work and writes NaN to the affected output rows;
 *     mla_get_status reports the flags.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID = -1,      /* bad argument (null pointer, shape, alignment)   */
    MLA_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. forced impl)     */
    MLA_ERR_BOUNDS = -3,       /* device flag: block id or length out of range     */
    MLA_ERR_WORKSPACE = -4,    /* workspace smaller than mla_workspace_bytes()     */
    MLA_ERR_CUDA = -5,         /* a CUDA launch or runtime call failed             */
    MLA_ERR_TIMEOUT = -6       /* device flag: a bounded wait gave up              */
} mla_status;

typedef enum {
    MLA_KV_BF16 = 0,           /* latent + rope key, bf16, one row per token       */
    MLA_KV_FP32 = 1,           /* latent + rope key, fp32, one row per token       */
    MLA_KV_INT2_ROT = 2,       /* rotated latent as grouped INT2 + bf16 rope key   */
    MLA_KV_INT2_ROT_QR = 3,    /* rotated latent and the (unrotated) rope key, both
                                  as grouped INT2: [c . R ; k_R] in (r + d_R) /
                                  group_size groups; d_R a multiple of group_size */
    MLA_KV_INT2_JOINT = 4      /* the whole row rotated by one eigenbasis R_j of
                                  [c ; k_R] ((r + d_R) x (r + d_R)) and stored as
                                  grouped INT2: [c ; k_R] . R_j in (r + d_R) /
                                  group_size groups; generic kernel only */
} mla_kv_kind;

typedef enum {
    MLA_IMPL_AUTO = 0,         /* tensor-core kernel where the shape allows it     */
    MLA_IMPL_SIMT = 1,         /* generic CUDA-core kernel, any supported shape    */
    MLA_IMPL_TCGEN05 = 2       /* tensor-core kernel; UNSUPPORTED if shape is not  */
} mla_impl;

/* Problem shape. All counts are element counts. */
typedef struct {
    int32_t num_heads;         /* H                                               */
    int32_t kv_lora_rank;      /* r, multiple of 8 (INT2: of group_size and 4)    */
    int32_t rope_dim;          /* d_R, multiple of 8 (may be 0 for FP32)          */
    int32_t v_head_dim;        /* d_v                                             */
    int32_t block_size;        /* tokens per cache block                          */
    int32_t num_blocks;        /* physical blocks in the pool                     */
    int32_t group_size;        /* INT2 group length along r (and d_R for
                                  INT2_ROT_QR / INT2_JOINT), a multiple of 4 in
                                  [4, 128], e.g. 32; else ignored                 */
    int32_t kind;              /* mla_kv_kind                                     */
    int32_t impl;              /* mla_impl                                        */
    int32_t num_splits_hint;   /* 0: planner's choice; k>0: aim for about k split-
                                  KV work units in total (1 = one per sequence)   */
    int32_t index_dim;         /* BF16 / FP32 kinds: elements of an extra per-token
                                  key stored after the rope key (e.g. a sparse-
                                  attention indexer key: 64 gives the 640-element
                                  row); a multiple of 8, <= 1024; 0 = none. INT2:
                                  must be 0. Attention never reads it.           */
    int32_t flags;             /* OR of mla_flag values; 0 for none               */
} mla_shape;

typedef enum {
    /* INT2_ROT / INT2_ROT_QR: the W_UV given to mla_decode / mla_verify is already
     * the folded W'_UV[h] = R^T . W_UV[h] of mla_fold_rotation, so the latent-space
     * output stays in the rotated basis and no o . R^T product is formed per call
     * (out = o_rot . R^T . W_UV[h] = o_rot . W'_UV[h]). */
    MLA_FLAG_WUV_FOLDED = 1,
    /* INT2_ROT / INT2_ROT_QR: the query's first r dims are already in the rotated
     * basis (q_lat . R, e.g. with R folded into the query's absorbed projection
     * once, as W_UV is folded by mla_fold_rotation), so the library does not rotate
     * the query; the rope dims are as always. With both flags set R is not read and
     * may be NULL. */
    MLA_FLAG_Q_ROTATED = 2
} mla_flag;

/* The paged cache. Block p, slot j is token row p*block_size + j.
 *   BF16/FP32:  latent     [num_blocks, block_size, r + d_R + index_dim]
 *                          (c, then k_R, then the optional extra key)
 *   INT2_ROT:   codes      [num_blocks, block_size, r / 4]    uint8, element e
 *                          of the row at bits 2*(e%4) of byte e/4
 *               scale_zero [num_blocks, block_size, r / group_size, 2] fp16
 *                          (scale, zero); value = fmaf(code, scale, zero)
 *               rope       [num_blocks, block_size, d_R]      bf16
 *   INT2_ROT_QR: codes      [num_blocks, block_size, (r + d_R) / 4] uint8 and
 *               scale_zero [num_blocks, block_size, (r + d_R) / group_size, 2]
 *                          fp16, as above over the row [c . R ; k_R]; rope unused
 *   INT2_JOINT: codes and scale_zero as INT2_ROT_QR, over the row [c ; k_R] . R_j
 * Unused members are NULL. */
typedef struct {
    void *latent;
    void *codes;
    void *scale_zero;
    void *rope;
} mla_cache;

/* Bytes of device workspace mla_decode / mla_verify need for B sequences with
 * q_len query rows each, on the current device. 0 on a bad shape. */
size_t mla_workspace_bytes(const mla_shape *shape, int32_t B, int32_t q_len);

/* Write new tokens into the paged cache (append / quantise).
 *   block_table [B, max_blocks_per_seq] int32: physical block of each logical
 *               block of each sequence.
 *   start_pos   [B] int32: position of the sequence's first new token.
 *   cu_new      [B + 1] int32: prefix sums of new-token counts; new tokens of
 *               sequence b are rows cu_new[b] .. cu_new[b+1]-1 of c_kv/k_rope.
 *   num_new     host int: cu_new[B] (total new tokens, sizes the launch).
 *   c_kv        [num_new, r]   bf16 (FP32 kind: fp32)
 *   k_rope      [num_new, d_R] bf16 (FP32 kind: fp32)
 *   R           INT2 kinds: [r, r] fp32 row-major, y = c . R (column j is the
 *               j-th eigenvector in ascending eigenvalue order); INT2_JOINT:
 *               [r + d_R, r + d_R], y = [c ; k_R] . R_j; else NULL.
 *   clip        INT2 kinds: [r / group_size] fp32 clip thresholds (INT2_ROT_QR:
 *               [(r + d_R) / group_size], the rope groups' after the latent's;
 *               INT2_JOINT: [(r + d_R) / group_size]); else NULL.
 *   status      optional [1] int32 device word; flags are OR-ed into it.
 * INT2 encoding per token and group g of group_size dims: y = fp32 fmaf chain
 * over k ascending; y clipped to [-clip[g], clip[g]]; scale =
 * fp16_rne((max - min) / 3), zero = fp16_rne(min); code = clamp(rint((y -
 * zero) / scale), 0, 3), 0 when scale == 0. INT2_ROT_QR: the rope groups encode
 * k_R as given (bf16 widened to fp32, not rotated) with their own thresholds.
 * INT2_JOINT: y = [c ; k_R] . R_j by the same fp32 chain over all r + d_R inputs.
 *   Source: OSCAR issue #10, maintainer reply (rotated + quantised latent in
 *   the cache, thresholds fit on the rotated latent). */
mla_status mla_latent_append(const mla_shape *shape, const mla_cache *cache,
                             const int32_t *block_table, int32_t max_blocks_per_seq,
                             int32_t B, const int32_t *start_pos, const int32_t *cu_new,
                             int32_t num_new, const void *c_kv, const void *k_rope,
                             const float *R, const float *clip, int32_t *status,
                             void *stream);

/* Decode attention, one query row per sequence (q_len = 1).
 *   seq_lens   [B] int32: tokens in the cache per sequence (>= 1).
 *   q          [B, 1, H, r + d_R] absorbed query, bf16 (FP32 kind: fp32).
 *   W_UV       [H, r, d_v] bf16 (FP32 kind: fp32).
 *   R          INT2 kinds: [r, r] fp32 (as in append; INT2_JOINT: [r + d_R,
 *              r + d_R], the query is rotated over all its dims and the output
 *              is (o_j . R_j^T)[0:r] before W_UV); else NULL. May be NULL with
 *              MLA_FLAG_WUV_FOLDED | MLA_FLAG_Q_ROTATED (not read).
 *   scale      softmax scale applied to q . k.
 *   out        [B, 1, H, d_v] bf16 (FP32 kind: fp32).
 *   lse        [B, 1, H] fp32, natural log of the softmax denominator.
 *   workspace  device scratch of at least mla_workspace_bytes(shape, B, 1).
 * The call is stream-ordered after prior work on `stream` (e.g. an append). */
mla_status mla_decode(const mla_shape *shape, const mla_cache *cache,
                      const int32_t *block_table, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens, int32_t B, const void *q,
                      const void *W_UV, const float *R, float scale, void *out,
                      float *lse, void *workspace, size_t workspace_bytes, void *stream);

/* Append then decode in one call: the same work and the same results as
 * mla_latent_append(shape, cache, block_table, max_blocks_per_seq, B, start_pos,
 * cu_new, num_new, c_kv, k_rope, R, clip, append_status, stream) followed by
 * mla_decode(shape, cache, block_table, max_blocks_per_seq, seq_lens, B, q, W_UV,
 * R, scale, out, lse, workspace, workspace_bytes, stream), every argument meaning
 * what it means there (seq_lens counts the appended tokens). For the bf16 and fp32
 * kinds the new tokens are copied by the launch that plans the decode, so the
 * copy adds no launch of its own to the step; for the INT2 kinds the append runs
 * as its own kernel first. Flags of the append (bad block or position) go to
 * append_status (may be NULL), those of the decode to the workspace
 * (mla_get_status). Argument errors of either part are returned before anything
 * is launched.
 *   Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10), the
 *   decode step of a serving loop: each step's new latent rows are cached, then
 *   the step's query attends over the whole cache. */
mla_status mla_append_decode(const mla_shape *shape, const mla_cache *cache,
                             const int32_t *block_table, int32_t max_blocks_per_seq, int32_t B,
                             const int32_t *start_pos, const int32_t *cu_new, int32_t num_new,
                             const void *c_kv, const void *k_rope, const float *clip,
                             int32_t *append_status, const int32_t *seq_lens, const void *q,
                             const void *W_UV, const float *R, float scale, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Speculative verify: q_len >= 1 draft rows per sequence, already appended, so
 * row i of sequence b sees positions 0 .. seq_lens[b] - q_len + i. Arguments as
 * mla_decode with q [B, q_len, H, r + d_R], out [B, q_len, H, d_v], lse
 * [B, q_len, H], workspace >= mla_workspace_bytes(shape, B, q_len).
 *   Source: "GLM-5.2 speculative drafting ..." (leyten/shard PR #5), TL;DR
 *   item 1 (drafts verified by the target); the causal window is this
 *   library's reading. */
mla_status mla_verify(const mla_shape *shape, const mla_cache *cache,
                      const int32_t *block_table, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens, int32_t B, int32_t q_len, const void *q,
                      const void *W_UV, const float *R, float scale, void *out,
                      float *lse, void *workspace, size_t workspace_bytes, void *stream);

/* mla_decode for callers that cannot allocate device memory at call time, such
 * as an inference-engine plugin whose enqueue step must not allocate, or a
 * serving process whose memory pool already holds the device's memory
 * (cudaMalloc can block, synchronise the device, or simply fail there). The
 * pages have no counterpart: this is a deployment convenience of the library.
 *   Arguments are those of mla_decode without the workspace; the caller still
 *   passes every input and output. Scratch comes from a fixed 32 MiB device
 *   array inside the library, held on every GPU that loads it until the
 *   process exits. No cudaMalloc, cudaFree or allocating library call is made.
 *   If the planner's default split count does not fit 32 MiB, fewer splits
 *   are used; if even one split per sequence does not fit (roughly B * q_len *
 *   H * kv_lora_rank * 4 bytes above 32 MiB), MLA_ERR_WORKSPACE is returned and
 *   nothing is launched.
 *   status: optional [1] int32 device word that receives this call's flag word
 *   (read it with mla_read_status_word); NULL to skip.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any stream capture. Calls
 *   outside capture look the address up again (cheap), so a module reload
 *   after cudaDeviceReset is followed; calls while `stream` is capturing use
 *   the address of the last call outside capture. Shape and implementation
 *   errors are those of mla_decode. Every call shares the one array: calls that can overlap on the
 *   GPU (other streams, other host threads) race on it and must be ordered by
 *   the caller. The flag word is reset at the start of each call; all other
 *   scratch is written before it is read. */
mla_status mla_decode_noalloc(const mla_shape *shape, const mla_cache *cache,
                              const int32_t *block_table, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, int32_t B, const void *q,
                              const void *W_UV, const float *R, float scale, void *out,
                              float *lse, int32_t *status, void *stream);

/* Wait for `stream`, read the device flags of the last decode/verify that used
 * `workspace` and return MLA_OK, MLA_ERR_BOUNDS or MLA_ERR_TIMEOUT. If
 * raw_flags is not NULL it receives the raw flag word (host int). */
mla_status mla_get_status(const void *workspace, int32_t *raw_flags, void *stream);

/* Read a device status word written by mla_latent_append (same meaning). */
mla_status mla_read_status_word(const int32_t *status, int32_t *raw_flags, void *stream);

/* Static description of a status code. */
const char *mla_status_string(mla_status status);

/* Which implementation mla_decode would run for this shape on the current
 * device (MLA_IMPL_SIMT or MLA_IMPL_TCGEN05), or a negative mla_status. */
int32_t mla_resolve_impl(const mla_shape *shape, int32_t q_len);

/* Diagnostics for benchmarking (host state, not thread-safe). While enabled,
 * every decode/verify call records a CUDA event pair on its stream around its
 * main attention kernel, and every entry point counts the kernels it launches.
 * mla_profile_enable(1) (re)starts the record; mla_profile_enable(2) does the same
 * but counts launches only (no event pairs between the kernels of a call);
 * mla_profile_enable(0) stops recording. mla_profile_read waits for the
 * recorded events and returns the summed duration of the attention kernels in
 * milliseconds, their launch count and the total kernel launch count (any
 * output pointer may be NULL). Events are created by the library on first use
 * (no device memory is allocated). */
mla_status mla_profile_enable(int32_t enable);
mla_status mla_profile_read(double *attention_ms, int32_t *attention_launches,
                            int32_t *kernel_launches);

/* Self-test of the device-side failure detection (diagnostic; no attention).
 * Launches one small kernel on `stream` that waits, with the same bounded
 * mbarrier wait the attention kernels use, on a barrier that nothing arrives on;
 * after `timeout_ns` the wait gives up, sets its CTA's abort flag and ORs the
 * timeout flag into the device word `status` (a caller-owned int32, zeroed by
 * the kernel first), and the kernel returns normally, leaving the context usable.
 * Read the outcome with mla_read_status_word (MLA_ERR_TIMEOUT expected).
 * timeout_ns must be in [1000, 100000000] (1 us .. 100 ms), else
 * MLA_ERR_INVALID; MLA_ERR_CUDA if the launch fails. */
mla_status mla_selftest_wait_timeout(uint64_t timeout_ns, int32_t *status, void *stream);

/* Write the extra per-token key (shape->index_dim elements, the caller's dtype:
 * bf16, or fp32 for the FP32 kind) of the tokens described exactly as for
 * mla_latent_append (block_table, start_pos, cu_new, num_new): index_key is
 * [num_new, index_dim] row-major, 16-byte aligned; it goes to elements
 * [r + d_R, r + d_R + index_dim) of each token's cache row. Errors as for
 * mla_latent_append; MLA_ERR_INVALID when index_dim is 0 or the kind is an INT2 one. */
mla_status mla_latent_append_index(const mla_shape *shape, const mla_cache *cache, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, int32_t B, const int32_t *start_pos,
                                   const int32_t *cu_new, int32_t num_new, const void *index_key,
                                   int32_t *status, void *stream);

/* Fold the output rotation of a rotated-INT2 layer into its up-projection, once
 * per layer: W_folded[h] = R^T . W_UV[h], i.e. W_folded[h][i][j] = sum_k R[k][i] *
 * W_UV[h][k][j], fp32 accumulation, rounded to bf16. Pass W_folded as W_UV with
 * MLA_FLAG_WUV_FOLDED set in shape->flags.
 *   Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
 *   maintainer reply: the up-projection runs on the dequantised latent, which the
 *   cache holds in the rotated basis, so its product with R^T can be taken ahead.
 *   shape  an INT2 kind (num_heads, kv_lora_rank, v_head_dim are read), else
 *          MLA_ERR_INVALID.
 *   R      [r, r] fp32 as in mla_latent_append.
 *   W_UV   [H, r, d_v] bf16.
 *   W_folded [H, r, d_v] bf16 output (must not alias W_UV). */
mla_status mla_fold_rotation(const mla_shape *shape, const float *R, const void *W_UV, void *W_folded,
                             void *stream);

/* ---- Calibration of the rotated-INT2 cache (once per layer, off the decode path).
 *   Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
 *   maintainer reply, "How the rotation adapts to the latent": Sigma = c^T c over
 *   calibration latents, its eigenvectors in ascending eigenvalue order (so that
 *   low-variance directions share INT2 groups) as R, clip thresholds fit on the
 *   rotated latent; and the "open refinement" paragraph after it, weighting latent
 *   directions by what the up-projection does with them (mla_calib_eigh_weighted).
 * Device calls are stream-ordered like the attention calls; host calls run on the
 * calling thread and touch no device. */
typedef enum { MLA_DTYPE_F64 = 0, MLA_DTYPE_F32 = 1, MLA_DTYPE_BF16 = 2 } mla_dtype;

/* sigma [d, d] fp64 (device) = X^T X, uncentred and unscaled, for calibration rows
 * X [n, d] (device, mla_dtype), accumulated in fp64. d <= 4096. */
mla_status mla_calib_covariance(const void *X, int64_t n, int32_t d, int32_t dtype, double *sigma, void *stream);

/* M [r, r] fp64 (device) = sum_h (W_UK[h]^T W_UK[h] + W_UV[h] W_UV[h]^T) for
 * W_UK [H, d_n, r] and W_UV [H, r, d_v] (device, both mla_dtype): how strongly each
 * latent direction reaches the keys and the values. */
mla_status mla_calib_projection_energy(const void *W_UK, const void *W_UV, int32_t H, int32_t d_n, int32_t r,
                                       int32_t d_v, int32_t dtype, double *M, void *stream);

/* HOST. Eigen-decomposition of the symmetric A [d, d] (host fp64; the lower triangle
 * is read): eigvals [d] ascending; the columns of R (R64 fp64 and/or R32 fp32
 * [d, d] row-major, either may be NULL) are the eigenvectors in that order, each
 * with its largest-magnitude entry (the first on ties) positive, so that y = c . R
 * as in mla_latent_append. MLA_ERR_UNSUPPORTED if the iteration fails to converge. */
mla_status mla_calib_eigh(const double *A, int32_t d, double *eigvals, double *R64, float *R32);

/* HOST. The up-projection-aware basis: as mla_calib_eigh for G = S^1/2 M S^1/2
 * (S^1/2 from the eigen-decomposition of S, negative eigenvalues taken as 0), with
 * S = mla_calib_covariance and M = mla_calib_projection_energy (host copies). With
 * M a multiple of the identity it is the basis of S itself. */
mla_status mla_calib_eigh_weighted(const double *S, const double *M, int32_t d, double *eigvals, double *R64,
                                   float *R32);

/* absY [n, d] fp64 (device) = |X . R| for calibration rows X [n, d] (device,
 * mla_dtype) and R [d, d] fp64 (device). */
mla_status mla_calib_project_abs(const void *X, int64_t n, int32_t d, int32_t dtype, const double *R, double *absY,
                                 void *stream);

/* HOST. Clip thresholds: clip[g] (fp32) = the pct-th percentile of absY[:, g*gs ..
 * g*gs + gs - 1] over all n rows, linearly interpolated between the two order
 * statistics around (n * gs - 1) * pct / 100. absY [n, d] host fp64 (e.g. a copy of
 * mla_calib_project_abs's output). d a multiple of group_size, 0 <= pct <= 100. */
mla_status mla_calib_thresholds(double *absY, int64_t n, int32_t d, int32_t group_size, double pct, float *clip);

/* Library ABI version (major * 100 + minor). */
int32_t mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
