/*
 * mla_b300.h -- C ABI of the B300 (sm_103a) absorbed, paged MLA decode path.
 *
 * What the path computes (Multi-head Latent Attention, DeepSeek-V2):
 *   "DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现"
 *   (PaperTrace) -- 2.1 joint KV down-projection and up-projection,
 *   2.2 matrix absorption at inference, 2.3 query compression,
 *   3.2 decoupled RoPE (score = content part in the latent space + position
 *   part), 3.3 the cached row c_KV | k_R.
 *   "DeepSeek R1的MLA：KV缓存的低秩压缩革命" -- 二 2.2 (precomputing
 *   Q W_uk^T), 五 item 4 (paged KV cache).
 *
 * One decode step, as the calls run on one stream:
 *   mla_append_latent  x W^DKV|W^KR, RoPE on k_R, store into the paged cache
 *   mla_project_q      [W^UQ|W^QR] (W^DQ x), RoPE on q_R
 *   mla_absorb_q       q_cat = [W^UK_h^T q_C,h | q_R,h]       (per head)
 *   mla_plan_decode    balanced split of all sequences' pages over the SMs
 *   mla_decode_attn    scores q_cat . [c | k_R], online softmax, latent output
 *   mla_combine        log-sum-exp merge of the split partial results
 *   mla_absorb_out     o_h = W^UV_h o_lat,h                    (per head)
 *   mla_combine_absorb_out  the two calls above as one
 *   mla_out_proj       u = W^O [o_1; ...; o_n_h]
 *
 * Conventions that hold for every call:
 *   - Every pointer argument except `dims` is DEVICE memory owned by the
 *     caller; the library never allocates, frees or keeps a pointer past the
 *     call. `dims` is host memory, read during the call only.
 *   - Every call only enqueues work on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream) and returns without waiting.
 *   - Weights use the column-vector convention W in R^{out x in}, stored
 *     row-major [out][in]; per-head blocks are consecutive rows.
 *   - Tensors are dense and row-major in the shapes given; element type is
 *     `dtype` (MLA_F32 = float, MLA_BF16 = bfloat16 bits) unless the
 *     signature says float.
 *   - Return value: MLA_OK, or an error found on the host before anything is
 *     enqueued (MLA_ERR_INVALID_ARG / UNSUPPORTED / WORKSPACE), or
 *     MLA_ERR_CUDA if a launch failed. mla_last_error() gives a message.
 *   - Errors found on the device (a block id outside the page pool, a
 *     position or length past the block table) cannot be returned: kernels
 *     OR a bit (MLA_DEV_*) into the caller's int32 `dev_status` word, skip
 *     the offending access, and carry on. Read the word after the stream
 *     has synchronised; `dev_status` may be NULL to skip the checks' report
 *     (the accesses are still skipped).
 */
#ifndef MLA_B300_H
#define MLA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 1

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size   */
  MLA_ERR_UNSUPPORTED = 2, /* shape/dtype this build has no kernel for      */
  MLA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required    */
  MLA_ERR_CUDA = 4         /* a CUDA launch or query failed                 */
} mla_status;

/* Bits kernels OR into *dev_status. */
#define MLA_DEV_BAD_BLOCK 0x1   /* block-table entry outside [0, num_pages)  */
#define MLA_DEV_BAD_POS 0x2     /* position outside the block table / RoPE   */
#define MLA_DEV_BAD_LEN 0x4     /* sequence length < 1 or past the table     */
#define MLA_DEV_TIMEOUT 0x8     /* a bounded wait inside a kernel gave up    */

typedef enum { MLA_F32 = 0, MLA_BF16 = 1, MLA_FP8_E4M3 = 2 } mla_dtype;

/* The FP8 latent cache (MLA_FP8_E4M3, decode only; DeepSeek-V2 MLA page 5.1
 * item 3 names quantizing the absorbed path): each cached row is
 *   bytes [0, d_c)               c_KV as E4M3 codes (OCP FP8, max 448)
 *   bytes [d_c, d_c + 2 d_r)     k_R as bf16 (the RoPE key is kept in bf16)
 *   bytes [d_c + 2 d_r, +4)      float scale s: c_KV[i] = e4m3(code[i]) * s
 *   then zeros up to MLA_FP8_ROW_BYTES (a multiple of 16).
 * The cache argument of mla_decode_attn is then [num_pages][page_size]
 * [MLA_FP8_ROW_BYTES(d_c, d_r)] bytes; q_cat is bf16, o_lat and lse float;
 * the plan and workspace are those of dtype MLA_FP8_E4M3. */
#define MLA_FP8_ROW_BYTES(d_c, d_r) ((((d_c) + 2 * (d_r) + 4) + 15) / 16 * 16)

/* Model dimensions (notation of the DeepSeek-V2 MLA page, 1.1 / 2.1 / 3.2). */
typedef struct {
  int n_h;       /* attention heads                                   */
  int d_h;       /* per-head no-PE query/key width                    */
  int d_r;       /* decoupled RoPE width d_h^R (even)                 */
  int d_c;       /* KV latent width                                   */
  int d_v;       /* per-head value width                              */
  int d_model;   /* hidden size d (append / project_q / out_proj)     */
  int d_cq;      /* query latent width d_c'; 0 = no query compression */
  int page_size; /* tokens per cache page                             */
} mla_dims;

/* Name of a status code; never NULL. */
const char* mla_status_string(int status);
/* Detail of the last non-OK status returned on this host thread. */
const char* mla_last_error(void);
int mla_abi_version(void);

/* RoPE table (RoFormer, which the MLA page's lineage section cites):
 * cos_sin[p][i] = {cos(p*theta_i), sin(p*theta_i)}, theta_i =
 * base^(-2i/d_r), for p < max_pos, i < d_r/2; computed in double, stored as
 * float [max_pos][d_r/2][2]. */
mla_status mla_rope_table(float* cos_sin, int max_pos, int d_r, double base, void* stream);

/* (a1) Append latent rows -- DeepSeek-V2 MLA page 2.1 (c_KV = W^DKV h) and
 * 3.2 (k_R = RoPE(W^KR h), cached beside c_KV, not compressed).
 *   x          [T][d_model]                 token hidden states
 *   w_dkv_kr   [d_c + d_r][d_model]         rows of W^DKV, then of W^KR
 *   seq_idx    [T] int32 or NULL            sequence of token t (NULL: t)
 *   pos        [T] int32                    position of token t
 *   block_table[B][max_pages] int32         physical page of each logical page
 *   rope       [max_pos][d_r/2][2] float    from mla_rope_table
 *   cache      [num_pages][page_size][d_c + d_r]   written at row
 *              (block_table[s][pos/page_size], pos%page_size); nothing else.
 * fp32 accumulation; the row is rounded once to `dtype` on store.
 * Device checks: seq_idx in [0,B), pos in [0, max_pages*page_size) and
 * < max_pos, block id in [0, num_pages). */
mla_status mla_append_latent(const void* x, const void* w_dkv_kr, const int32_t* seq_idx,
                             const int32_t* pos, const int32_t* block_table, int B,
                             int max_pages, int num_pages, int T, const float* rope,
                             int max_pos, void* cache, mla_dtype dtype, const mla_dims* dims,
                             int32_t* dev_status, void* stream);

/* (a2) Query projection -- DeepSeek-V2 MLA page 2.3 (c_Q = W^DQ h,
 * q_C = W^UQ c_Q) and 3.2 (q_R = RoPE(W^QR c_Q), one slice per head).
 *   x        [T][d_model]
 *   w_dq     [d_cq][d_model], or NULL when dims->d_cq == 0 (then c_Q = x)
 *   w_uq_qr  [n_h][d_h + d_r][K], K = d_cq or d_model: per head the rows of
 *            W^UQ_h then of W^QR_h
 *   pos      [T] int32, rope as for mla_append_latent
 *   c_q      [T][d_cq] scratch the caller provides (ignored if d_cq == 0)
 *   q        [T][n_h][d_h + d_r] output: [q_C,h | RoPE(q_R,h)]
 * fp32 accumulation; c_q and q are stored in `dtype`. */
mla_status mla_project_q(const void* x, const void* w_dq, const void* w_uq_qr,
                         const int32_t* pos, int T, const float* rope, int max_pos,
                         void* c_q, void* q, mla_dtype dtype, const mla_dims* dims,
                         int32_t* dev_status, void* stream);

/* (a3) Absorb W^UK into the query -- DeepSeek-V2 MLA page 2.2
 * (q^T W^UK c = (W^UK^T q)^T c); R1 MLA page 二 2.2 (precompute Q W_uk^T).
 *   q      [B][n_h][d_h + d_r]
 *   w_uk   [n_h*d_h][d_c]           (W^UK, head h = rows h*d_h ..)
 *   q_cat  [B][n_h][d_c + d_r]      output: [W^UK_h^T q_C,h | q_R,h]
 * fp32 accumulation, one rounding to `dtype`. */
mla_status mla_absorb_q(const void* q, const void* w_uk, void* q_cat, int B, mla_dtype dtype,
                        const mla_dims* dims, void* stream);

/* (a4) Split plan. The pages of all sequences, in order, are cut into
 * contiguous ranges of near-equal cost, one per worker (an SM or SM pair of
 * the decode kernel the same dtype/dims select). Cost: one unit per page,
 * plus, on the tcgen05 path, 4 units per sequence a worker starts (its
 * fixed cost of fetching Q and writing O), so a worker that starts a new
 * sequence takes fewer pages. A sequence cut into k > 1 ranges gets k
 * partial results that mla_combine merges. The plan lives in `workspace`
 * and depends only on seq_lens, B, dtype, dims and the device.
 *   seq_lens [B] int32 (>= 1; tokens already in the cache, including the
 *            one being decoded). */
size_t mla_decode_workspace_size(int B, mla_dtype dtype, const mla_dims* dims);
mla_status mla_plan_decode(const int32_t* seq_lens, int B, int max_pages, void* workspace,
                           size_t ws_bytes, mla_dtype dtype, const mla_dims* dims,
                           int32_t* dev_status, void* stream);

/* (a5) Paged split-KV decode attention in the latent space -- DeepSeek-V2
 * MLA page 3.2: s_j = (q_abs . c_j + q_R . k_R,j) * softmax_scale over the
 * sequence's cached tokens j < seq_lens[b]; softmax; o_lat = sum_j p_j c_j.
 *   q_cat   [B][n_h][d_c + d_r]        from mla_absorb_q
 *   cache   [num_pages][page_size][d_c + d_r]
 *   block_table [B][max_pages] int32, seq_lens [B] int32
 *   workspace   planned by mla_plan_decode with the same seq_lens
 *   o_lat   [B][n_h][d_c] float, lse [B][n_h] float (natural log of
 *           sum_j exp(s_j)): written for sequences the plan does not split;
 *           split sequences are written by mla_combine.
 * bf16 path: bf16 tensor-core products with fp32 accumulation; probabilities
 * are rounded to bf16 before the P.V product. f32 path: fp32 throughout. */
mla_status mla_decode_attn(const void* q_cat, const void* cache, const int32_t* block_table,
                           int max_pages, int num_pages, const int32_t* seq_lens, int B,
                           float softmax_scale, void* workspace, size_t ws_bytes, float* o_lat,
                           float* lse, mla_dtype dtype, const mla_dims* dims,
                           int32_t* dev_status, void* stream);

/* (a5, several new tokens) Decode of q_len new tokens per sequence at once
 * -- multi-token prediction and speculative drafts, DeepSeek-V2 MLA page 4.3
 * and 6 (MLA combined with MTP). The q_len tokens of sequence b already sit
 * at the last q_len of its seq_lens[b] cached positions (appended before
 * the call), and new token t sees every cached position up to and
 * including its own: seq_lens[b] - q_len + 1 + t of them. Query row
 * v = b * q_len + t.
 *   q_cat  [B][q_len][n_h][d_c + d_r]; o_lat [B][q_len][n_h][d_c] float;
 *   lse    [B][q_len][n_h] float; the other arguments as for
 *          mla_decode_attn, the workspace sized by
 *          mla_decode_workspace_size(B * q_len, ...) and planned by
 *          mla_plan_decode_mtp with the same seq_lens and q_len.
 * Rows whose sequence the plan splits are finished by
 * mla_combine(workspace, ws_bytes, B * q_len, ...); mla_absorb_q and
 * mla_absorb_out take the B * q_len query rows as their batch.
 * 1 <= q_len <= MLA_MAX_NEW_TOKENS; seq_lens[b] >= q_len (a shorter one is
 * reported as MLA_DEV_BAD_LEN for the rows that would see no token). The
 * query rows of one sequence sit next to each other in the plan, so the
 * SMs that read the same pages run at about the same time and the second
 * read of a page is served by L2. */
#define MLA_MAX_NEW_TOKENS 8
mla_status mla_plan_decode_mtp(const int32_t* seq_lens, int B, int q_len, int max_pages,
                               void* workspace, size_t ws_bytes, mla_dtype dtype,
                               const mla_dims* dims, int32_t* dev_status, void* stream);
mla_status mla_decode_attn_mtp(const void* q_cat, const void* cache, const int32_t* block_table,
                               int max_pages, int num_pages, const int32_t* seq_lens, int B,
                               int q_len, float softmax_scale, void* workspace, size_t ws_bytes,
                               float* o_lat, float* lse, mla_dtype dtype, const mla_dims* dims,
                               int32_t* dev_status, void* stream);

/* (a6) Merge split partials: lse = log sum_s exp(lse_s),
 * o_lat = sum_s exp(lse_s - lse) o_s, for every sequence the plan split. */
mla_status mla_combine(const void* workspace, size_t ws_bytes, int B, float* o_lat, float* lse,
                       mla_dtype dtype, const mla_dims* dims, void* stream);

/* (a7) Map the latent output back per head -- DeepSeek-V2 MLA page 2.2
 * (the W^UV half of W~^O = W^O W^UV, applied unfused).
 *   o_lat [B][n_h][d_c] float; w_uv [n_h*d_v][d_c] in `dtype`;
 *   o     [B][n_h*d_v] in `out_dtype`. fp32 accumulation. */
mla_status mla_absorb_out(const float* o_lat, const void* w_uv, void* o, int B, mla_dtype dtype,
                          mla_dtype out_dtype, const mla_dims* dims, void* stream);

/* (a6 + a7) mla_combine followed by mla_absorb_out, as one call: the merge
 * of each split sequence's partials feeds the W^UV product directly. Writes
 * o_lat and lse exactly as mla_combine does (bit for bit) and o exactly as
 * mla_absorb_out does. Arguments as for those two calls; `workspace` holds
 * the plan and partials of the preceding mla_decode_attn. On shapes without
 * a fused kernel it runs the two kernels one after the other. */
mla_status mla_combine_absorb_out(const void* workspace, size_t ws_bytes, int B, float* o_lat,
                                  float* lse, const void* w_uv, void* o, mla_dtype dtype,
                                  mla_dtype out_dtype, const mla_dims* dims, int32_t* dev_status,
                                  void* stream);

/* (a8) Output projection u = W^O [o_1; ...; o_n_h] -- DeepSeek-V2 MLA
 * page 2.2 (W^O).
 *   o [B][n_h*d_v] in `dtype`; w_o [d_model][n_h*d_v] in `dtype`;
 *   u [B][d_model] float. fp32 accumulation. */
mla_status mla_out_proj(const void* o, const void* w_o, float* u, int B, mla_dtype dtype,
                        const mla_dims* dims, void* stream);

/* Prefill in the MHA form -- "kv-cache 的优化学习" (cnblogs), closing
 * note: the cache holds the MLA form; a prompt is expanded to per-head keys
 * and values (MHA) for prefill and decoding stays in the latent form; the
 * DeepSeek-V2 MLA page 2.1 gives the expansion k^C = W^UK c, v^C = W^UV c and
 * 3.2 the key [k^C_h ; k^R] with the RoPE key shared by all heads. For one
 * sequence of N prompt tokens already appended to the cache:
 *   mla_gather_latent   rows [N][d_c + d_r] = the cache rows of positions
 *                       0..N-1 of sequence `seq` (dense copy).
 *   mla_expand_kv       k_nope [N][n_h][d_h] = c W^UK_h^T and
 *                       v [N][n_h][d_v] = c W^UV_h^T for every head (c =
 *                       rows[:, :d_c]); fp32 accumulation, stored in `dtype`.
 *   mla_prefill_attn    o [N][n_h][d_v] (bf16) and lse [N][n_h] (float, may
 *                       be NULL): token i attends to tokens j <= i,
 *                       s_j = (q_i,h . [k_nope_j,h ; k_R,j]) * softmax_scale,
 *                       with q [N][n_h][d_h + d_r] from mla_project_q (T = N).
 *                       bf16 tensor-core products, fp32 accumulation and
 *                       softmax, probabilities rounded to bf16 for P.V.
 *                       Built for bf16 with n_h = 128, d_h = d_v = 128,
 *                       d_r = 64, d_c = 512 (else MLA_ERR_UNSUPPORTED). */
mla_status mla_gather_latent(const void* cache, const int32_t* block_table, int max_pages,
                             int num_pages, int seq, int n_tokens, void* rows, mla_dtype dtype,
                             const mla_dims* dims, int32_t* dev_status, void* stream);
mla_status mla_expand_kv(const void* rows, const void* w_uk, const void* w_uv, void* k_nope,
                         void* v, int n_tokens, mla_dtype dtype, const mla_dims* dims,
                         void* stream);
mla_status mla_prefill_attn(const void* q, const void* k_nope, const void* rows, const void* v,
                            void* o, float* lse, int n_tokens, float softmax_scale,
                            mla_dtype dtype, const mla_dims* dims, int32_t* dev_status,
                            void* stream);

/* Fused absorption -- DeepSeek-V2 MLA page 2.2, the form that folds the
 * up-projections into the neighbouring weights once, ahead of decoding:
 * W~^Q = W^UQ^T W^UK (query side) and W~^O = W^O W^UV (output side). The
 * per-head calls above (mla_absorb_q / mla_absorb_out) apply W^UK and W^UV
 * unfused instead; these calls are the alternative, measured against it.
 *
 * mla_fuse_query_weights: w_uq_qr [n_h][d_h + d_r][K] (as for
 *   mla_project_q, K = d_cq or d_model), w_uk [n_h*d_h][d_c] ->
 *   w_fused_q [n_h][d_c + d_r][K]: per head the d_c rows of
 *   W^UK_h^T W^UQ_h, then the d_r rows of W^QR_h unchanged. fp32
 *   accumulation, one rounding to `dtype`.
 * mla_project_q_absorbed: mla_project_q with w_fused_q in place of w_uq_qr:
 *   writes q_cat [T][n_h][d_c + d_r] (RoPE on its last d_r columns)
 *   directly, so no mla_absorb_q follows.
 * mla_fuse_output_weights: w_o [d_model][n_h*d_v], w_uv [n_h*d_v][d_c] ->
 *   w_fused_o [d_model][n_h*d_c] = the per-head products W^O_h W^UV_h side
 *   by side. fp32 accumulation, one rounding to `dtype`.
 * mla_out_proj_absorbed: u [B][d_model] float = w_fused_o . o_lat (o_lat
 *   [B][n_h][d_c] float, flattened per row); for bf16 weights o_lat is first
 *   rounded to bf16 into the caller's scratch o_lat_lowp [B][n_h*d_c]
 *   (ignored for fp32). Replaces mla_absorb_out + mla_out_proj.
 * The fused weights are larger: (d_c + d_r) K per head instead of
 * (d_h + d_r) K + d_h d_c, and d_model n_h d_c instead of
 * n_h d_v (d_model + d_c). */
mla_status mla_fuse_query_weights(const void* w_uq_qr, const void* w_uk, void* w_fused_q,
                                  mla_dtype dtype, const mla_dims* dims, void* stream);
mla_status mla_project_q_absorbed(const void* x, const void* w_dq, const void* w_fused_q,
                                  const int32_t* pos, int T, const float* rope, int max_pos,
                                  void* c_q, void* q_cat, mla_dtype dtype, const mla_dims* dims,
                                  int32_t* dev_status, void* stream);
mla_status mla_fuse_output_weights(const void* w_o, const void* w_uv, void* w_fused_o,
                                   mla_dtype dtype, const mla_dims* dims, void* stream);
mla_status mla_out_proj_absorbed(const float* o_lat, void* o_lat_lowp, const void* w_fused_o,
                                 float* u, int B, mla_dtype dtype, const mla_dims* dims,
                                 void* stream);

/* Allocation-free decode (the paper has no counterpart: this is a service
 * for callers, not a step of the method). Some callers cannot allocate
 * device memory when they decode -- plugin hosts and embedded runtimes that
 * hand over a stream but no allocator; serving loops that ban device
 * allocations after start-up so no step blocks on the allocator -- and so
 * cannot supply the workspace mla_decode_attn needs. This call runs the same
 * plan -> decode -> combine sequence with that workspace held in a
 * file-scope device array of MLA_STATIC_SCRATCH_BYTES, which every GPU that
 * loads this library keeps until the process exits. It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *   Arguments, checks and outputs are those of mla_decode_attn (o_lat and
 *   lse are final for every sequence; no mla_combine call follows).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   Every call uses the same array and leaves its contents behind; nothing
 *   in it has to start at zero. Calls that overlap on the GPU (other
 *   streams, other host threads) race on it -- serialise them.
 *   A batch whose plan and partials need more than MLA_STATIC_SCRATCH_BYTES
 *   (see mla_decode_workspace_size) is refused with MLA_ERR_WORKSPACE before
 *   anything is enqueued. */
#define MLA_STATIC_SCRATCH_BYTES (48u << 20)
mla_status mla_decode_attn_static(const void* q_cat, const void* cache,
                                  const int32_t* block_table, int max_pages, int num_pages,
                                  const int32_t* seq_lens, int B, float softmax_scale,
                                  float* o_lat, float* lse, mla_dtype dtype,
                                  const mla_dims* dims, int32_t* dev_status, void* stream);

/* Decode on the FP8 latent cache through the bf16 decode kernels
 * (DeepSeek-V2 MLA page 5.1 item 3: the absorbed path kept on a quantized
 * cache). The call widens every page the batch reads into bf16 rows
 * (c_KV[i] = bf16(e4m3(code[i]) * s), k_R copied) in the workspace, under an
 * identity block table, then plans, decodes and combines those rows exactly
 * as mla_decode_attn with dtype MLA_BF16 does (the tcgen05 kernel wherever
 * it supports the shape). o_lat and lse are final; no mla_combine follows.
 *   q_cat      [B][n_h][d_c + d_r] bf16, device.
 *   cache      [num_pages][page_size][MLA_FP8_ROW_BYTES(d_c, d_r)] bytes in
 *              the FP8 row format above, device, 16-byte aligned.
 *   block_table, max_pages, num_pages, seq_lens, B, softmax_scale, o_lat,
 *              lse, dev_status, stream: as mla_decode_attn.
 *   workspace  >= mla_decode_fp8_staged_workspace_size(B, max_pages, dims)
 *              bytes of device memory, 256-byte aligned, owned by the
 *              caller; nothing in it has to start at zero. It holds the
 *              bf16 plan and partials, the identity table and
 *              B * max_pages * page_size * (d_c + d_r) bf16 rows.
 * Errors: as mla_decode_attn; MLA_ERR_UNSUPPORTED for B > 65535 or d_r not
 * a multiple of 8; MLA_ERR_INVALID_ARG for a cache not 16-byte aligned or a
 * workspace not 256-byte aligned. Block ids outside [0, num_pages) are reported through
 * dev_status (MLA_DEV_BAD_BLOCK) and read as zero rows. The workspace size
 * depends on the decode kernel the device selects; query it under the same
 * mla_force_decode_path setting as the call. */
size_t mla_decode_fp8_staged_workspace_size(int B, int max_pages, const mla_dims* dims);
mla_status mla_decode_attn_fp8_staged(const void* q_cat, const void* cache,
                                      const int32_t* block_table, int max_pages, int num_pages,
                                      const int32_t* seq_lens, int B, float softmax_scale,
                                      void* workspace, size_t ws_bytes, float* o_lat, float* lse,
                                      const mla_dims* dims, int32_t* dev_status, void* stream);

/* Diagnostic for the tensor-core decode kernel's data path (no counterpart
 * in the method): one 64-token page through the same tcgen05 operand
 * layouts, without softmax. All bf16 row-major device tensors:
 *   q_cat [128][576], page [64][576], pmat [128][64];
 *   s_out [128][64]  float = q_cat . page^T;
 *   o_out [128][256] float = pmat . page[:, 256*half : 256*half + 256].
 * Returns MLA_ERR_UNSUPPORTED on a device without the sm_103 tensor-core
 * kernels. */
mla_status mla_tc_selftest(const void* q_cat, const void* page, const void* pmat, float* s_out,
                           float* o_out, int half, int32_t* dev_status, void* stream);

/* Which decode kernel the given dtype/dims select on the current device:
 * 1 = tcgen05 tensor-core kernel (each SM of a pair owns half of d_c),
 * 2 = the older tcgen05 score/value pair kernel (only when forced),
 * 0 = CUDA-core (SIMT) kernel. */
int mla_decode_path(mla_dtype dtype, const mla_dims* dims);

/* Pin the decode kernel choice for this process: 0 = always the SIMT kernel
 * (and the CUDA-core GEMMs), 1 = the tcgen05 kernels wherever they support
 * the shape, 2 = as 1 but the score/value pair decode kernel, -1 =
 * automatic (default, same as 1). Plans, workspaces and decode calls must be
 * made under the same setting. Used to cross-check the kernels against each
 * other. */
void mla_force_decode_path(int path);

#ifdef __cplusplus
}
#endif
#endif /* MLA_B300_H */
