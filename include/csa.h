/*
 * csa.h — C ABI of libcsa, the Compressed Sparse Attention (CSA) hot path on one GPU.
 *
 * The operations are those of the CSA layer described in "DeepSeek V4-Flash: The Cost of
 * Deciding What to Read" (sections "The compressor has two streams and they overlap",
 * "The Lightning Indexer", "Attention sink, and heads that abstain", "The sliding window
 * is not an optimisation", "Key and value are the same vector") and of its CSA2 variant
 * in "DeepSeek-V4.1-Flash's KV-Cache Compression, Checked Down to the Byte", section 3
 * (Full / Reindex / Reuse modes, Hierarchical Sparse Indexer).
 *
 * Conventions (every call):
 *  - All tensor arguments are DEVICE pointers to caller-owned memory, dense row-major in the
 *    shapes given, 16-byte aligned.  The library allocates nothing; scratch comes from the
 *    caller's workspace `ws` of at least csa_workspace_size(...) bytes (16-byte aligned).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and returns a csa_status.  Arguments are validated on the host before any launch; on a
 *    validation error nothing is launched.  CSA_ERR_CUDA reports a failed launch.
 *  - Errors the kernels detect on the device (a bounded wait that expired, an index out of
 *    range) are recorded in a device error word; csa_get_last_error() synchronises the
 *    stream, returns and clears it.
 *  - No C++ exceptions cross this boundary; no torch types appear in it.
 *  - Shapes use: B sequences, T query tokens per sequence, H query heads, d head dim,
 *    HI indexer heads, dI indexer dim, m compression ratio, k top-k, W window,
 *    E_cap rows allocated per sequence in the compressed caches.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa_stream_t; /* same object as cudaStream_t */

typedef enum {
  CSA_OK = 0,
  CSA_ERR_NULL = 1,        /* a required pointer is NULL                                   */
  CSA_ERR_SHAPE = 2,       /* a size is out of range or inconsistent                       */
  CSA_ERR_DTYPE = 3,       /* unsupported dtype combination                                */
  CSA_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned                             */
  CSA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than csa_workspace_size()       */
  CSA_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed                         */
  CSA_ERR_TIMEOUT = 7,     /* a device-side bounded wait expired (pipeline stalled)        */
  CSA_ERR_INDEX = 8        /* a selected index was >= E_cap (the row was skipped)          */
} csa_status;

/* CSA_MXFP4 is a storage format of indexer keys only (csa_config.kidx, csa_compress_kv's
 * out_dtype): per key of 128 channels, 64 payload bytes of E2M1 codes (channel 2i in the low
 * nibble of byte i) and, in a separate array, 4 UE8M0 scale bytes (byte j for channels
 * 32j .. 32j+31, value 2^(byte - 127)) kept as one little-endian 32-bit word: 68 bytes a key
 * (V4.1 diagram, byte ledger "Single request / logical serving KV storage": "Indexer K:
 * 128 channels, MXFP4, 64 packed bytes + 4 UE8M0 scales"). */
typedef enum { CSA_F32 = 0, CSA_BF16 = 1, CSA_E4M3 = 2, CSA_MXFP4 = 3 } csa_dtype;

typedef struct {
  int32_t B, H, d;      /* sequences, query heads, head dim (= compressed entry dim)        */
  int32_t HI, dI;       /* indexer heads, indexer dim                                       */
  int32_t m;            /* compression ratio (1 = CSA2 one-to-one store)                    */
  int32_t k;            /* entries kept by the top-k                                        */
  int32_t W;            /* sliding-window length                                            */
  csa_dtype act;        /* CSA_F32 or CSA_BF16: q, qI, KV streams, caches, window, output   */
  csa_dtype kidx;       /* indexer keys: == act, CSA_E4M3 (+ fp32 row scale), or CSA_MXFP4
                           (act == CSA_BF16, dI == 128, HI 32 or 64; E_cap % 4 == 0)       */
  float softmax_scale;  /* attention logit scale, e.g. 1/sqrt(d)                            */
} csa_config;

/* Operation ids for csa_workspace_size. */
typedef enum {
  CSA_OP_COMPRESS = 0, CSA_OP_INDEXER = 1, CSA_OP_TOPK = 2, CSA_OP_ATTN = 3,
  CSA_OP_DECODE = 4, CSA_OP_POOL = 5, CSA_OP_INDEXER_TOPK = 6, CSA_OP_DENSE_ATTN = 7,
  CSA_OP_HCA_DECODE = 8, CSA_OP_TOPK_BF16 = 9, CSA_OP_INDEXER_TOPK_BF16 = 10
} csa_op;

/*
 * csa_workspace_size — bytes of scratch the operation needs.
 *   rows   : query rows (B*T) of the call;
 *   n_cols : the longest score row (E_cap, or n_cand) for TOPK / DECODE / INDEXER_TOPK;
 *            T (queries per sequence) for ATTN and INDEXER; E_cap for DENSE_ATTN and
 *            HCA_DECODE (rows = B*T, and B for HCA_DECODE).  (POOL: see
 *            csa_block_pool_workspace_size.)
 * Returns 0 for operations that need none, (size_t)-1 for an invalid configuration.
 */
size_t csa_workspace_size(csa_op op, const csa_config *cfg, int64_t rows, int64_t n_cols);

/*
 * csa_compress_kv — gated two-stream compression ("The compressor has two streams and
 * they overlap"): entry i mixes stream a over tokens [m*i, m*(i+1)) and stream b over
 * [m*(i-1), m*i) with a per-channel softmax of the 2m logits Z + B (m logits for entry 0,
 * which has no previous block), then sums the matching C values with those weights.
 *
 *   dim        : channels (d for the main KV, dI for indexer keys)
 *   kv, z      : [B, n_tok, 2, dim] (cfg->act) — C^a/C^b and Z^a/Z^b of tokens
 *                tok0 .. tok0+n_tok-1; [..][0][..] is stream a, [..][1][..] stream b
 *   bias       : [2, m, dim] fp32 — B^a, B^b by position inside the block
 *   ent_begin, ent_end : entries to produce; needs tok0 <= m*max(ent_begin-1, 0) and
 *                m*ent_end <= tok0 + n_tok (else CSA_ERR_SHAPE)
 *   out        : [B, E_cap, dim] in out_dtype (CSA_F32, CSA_BF16 or CSA_E4M3), or
 *                [B, E_cap, dim/2] E2M1 payload bytes for CSA_MXFP4 (dim == 128); entry i is
 *                written at row i, rows outside [ent_begin, ent_end) are untouched
 *   out_scale  : CSA_E4M3: [B, E_cap] fp32 (scale = amax/448, code = e4m3_rn_satfinite(x /
 *                scale); an all-zero row gets scale 1).  CSA_MXFP4: [B, E_cap] 32-bit words of
 *                4 UE8M0 bytes, per 32 channels X = 2^(floor(log2(amax)) - 2) (the OCP MX
 *                rule; exponent clamped to [-127, 127], an all-zero block gets 2^-127) and
 *                code = nearest E2M1 value of x / X (ties to even, saturating at 6, sign kept).
 *                Required iff out_dtype is one of the two; 16-byte aligned.
 */
csa_status csa_compress_kv(const csa_config *cfg, int32_t dim, const void *kv, const void *z,
                           const float *bias, int64_t n_tok, int64_t tok0, int64_t ent_begin,
                           int64_t ent_end, void *out, csa_dtype out_dtype, void *out_scale,
                           int64_t E_cap, csa_stream_t stream);

/*
 * csa_compress_kv_single — one-stream compression without overlap: HCA ("Heavily
 * Compressed Attention": the compressor at m' = 128 with a single KV stream) and the CSA2
 * encoder (V4.1 diagram, "Encoder groups compress pairs": m = 2, channel-wise softmax per
 * pair, no positional embedding).  With m = cfg->m, entry i of every channel c is
 *   sum_j softmax_j(Z[m*i + j, c] + bias[j, c]) * C[m*i + j, c],   j = 0 .. m-1
 * (bias NULL: no positional term).  Only cfg->B, cfg->m and cfg->act are read.
 *
 *   dim        : channels, even, 2 .. 4096
 *   kv, z      : [B, n_tok, dim] (cfg->act) — C and Z of tokens tok0 .. tok0+n_tok-1
 *   bias       : [m, dim] fp32 or NULL
 *   ent_begin, ent_end : entries to produce; needs tok0 <= m*ent_begin and
 *                m*ent_end <= tok0 + n_tok (else CSA_ERR_SHAPE)
 *   out        : [B, E_cap, dim] (cfg->act); rows outside [ent_begin, ent_end) untouched
 */
csa_status csa_compress_kv_single(const csa_config *cfg, int32_t dim, const void *kv, const void *z,
                                  const float *bias, int64_t n_tok, int64_t tok0, int64_t ent_begin,
                                  int64_t ent_end, void *out, int64_t E_cap, csa_stream_t stream);

/*
 * csa_indexer_scores — lightning-indexer scores ("The Lightning Indexer"):
 *   score[r, s] = sum_h w[r, h] * ReLU(qI[r, h, :] . kI[b, s, :])      (kI dequantised)
 * for query row r = b*T + t at position q_pos[r], over entries s < nv = min(floor((q_pos+1)/m),
 * E_cap) — the causal rule of "The sliding window is not an optimisation"; every other
 * column of the row is set to -inf.
 *
 *   qI     : [B, T, HI, dI] (cfg->act);  w : [B, T, HI] fp32;  q_pos : [B*T] int64
 *   kI     : [B, E_cap, dI] in cfg->kidx ([B, E_cap, 64] payload bytes for CSA_MXFP4, 32-byte
 *            aligned); kscale : [B, E_cap] fp32 iff kidx == CSA_E4M3, [B, E_cap] 32-bit
 *            UE8M0 scale words iff kidx == CSA_MXFP4 (see csa_dtype), else NULL
 *   cand   : NULL — score every column s in [0, n_cols) with n_cols = E_cap;
 *            else [B*T, n_cand] int32 positions (CSA2 Reindex: a candidate pool); column j
 *            scores position cand[r, j]; cand < 0 or >= nv gives -inf.
 *   scores : [B*T, ld_scores] fp32, ld_scores >= n_cols (E_cap or n_cand)
 * bf16 keys with dI == 128 run on the tcgen05 tensor cores (fp32 accumulate); E4M3 keys run
 * the FP8 tensor-core path with qI split into two E4M3 terms; MXFP4 keys run the block-scaled
 * tensor-core path (E2M1 keys x the two E4M3 query terms, the keys' UE8M0 scales applied by
 * the MMA; "FP4, down to the index scores"); otherwise a CUDA-core path.
 */
csa_status csa_indexer_scores(const csa_config *cfg, const void *qI, const float *w, int32_t T,
                              const int64_t *q_pos, const void *kI, const void *kscale,
                              int64_t E_cap, const int32_t *cand, int32_t n_cand, float *scores,
                              int64_t ld_scores, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_indexer_scores_bf16 — csa_indexer_scores writing each score rounded to BF16 (round to
 * nearest even of the fp32 score csa_indexer_scores writes; -inf as BF16 -inf): scores is
 * [B*T, ld_scores] 16-bit ("FP4, down to the index scores": the index scores in BF16 before
 * the top-k selector).  Same arguments, workspace and errors.
 */
csa_status csa_indexer_scores_bf16(const csa_config *cfg, const void *qI, const float *w, int32_t T,
                                   const int64_t *q_pos, const void *kI, const void *kscale,
                                   int64_t E_cap, const int32_t *cand, int32_t n_cand, void *scores,
                                   int64_t ld_scores, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_indexer_topk — csa_indexer_scores followed by csa_topk over each row's visible entries
 * ("The Lightning Indexer": keep the k best; ties to the lowest position) in one call:
 * idx[r, 0:k] holds the k best visible positions of query row r in ascending order, -1
 * padded, exactly as csa_topk returns them from the scores csa_indexer_scores writes.
 *
 *   qI, w, T, q_pos, kI, kscale, E_cap : as in csa_indexer_scores (all entries, no candidates)
 *   idx : [B*T, cfg->k] int32
 *   ws  : csa_workspace_size(CSA_OP_INDEXER_TOPK, cfg, B*T, E_cap) bytes
 * The scores live in ws (the caller holds no score matrix) and the same kernels as the two
 * separate calls run on them.
 */
csa_status csa_indexer_topk(const csa_config *cfg, const void *qI, const float *w, int32_t T,
                            const int64_t *q_pos, const void *kI, const void *kscale, int64_t E_cap,
                            int32_t *idx, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_indexer_topk_bf16 — csa_indexer_topk over BF16 scores: idx is exactly what
 * csa_topk_bf16 returns on the scores csa_indexer_scores_bf16 writes (the scores, 2 bytes
 * each, live in ws).  ws : csa_workspace_size(CSA_OP_INDEXER_TOPK_BF16, cfg, B*T, E_cap).
 */
csa_status csa_indexer_topk_bf16(const csa_config *cfg, const void *qI, const float *w, int32_t T,
                                 const int64_t *q_pos, const void *kI, const void *kscale, int64_t E_cap,
                                 int32_t *idx, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_topk — per row, the cfg->k best of scores[r, 0:n_valid[r]] under the total order
 * (score descending, position ascending; -0 == +0), written to idx[r, 0:k] in ascending
 * position order, padded with -1 when fewer than k are valid.  Deterministic.
 *
 *   scores  : [rows, ld] fp32;  n_valid : [rows] int32 (NULL = n_cols for every row)
 *   cand    : NULL, or [rows, ld_cand = n_cols] int32 ascending positions, optionally followed by
 *             -1 padding (slots from the first -1 on are not candidates): idx holds cand[r, j]
 *             instead of the column j (CSA2 Reindex over a pool)
 *   idx     : [rows, k] int32
 */
csa_status csa_topk(const csa_config *cfg, const float *scores, int64_t ld, int64_t rows,
                    int64_t n_cols, const int32_t *n_valid, const int32_t *cand, int32_t *idx,
                    void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_topk_bf16 — csa_topk over BF16 scores ([rows, ld] 16-bit): the same total order on the
 * BF16 values (score descending, position ascending; -0 == +0), output ascending, -1 padded.
 * BF16 rounding makes many scores equal; ties go to the lowest position.  Rows of any length
 * run the one-CTA-per-row or the histogram path (a 12-bit digit of the 16-bit key, then one
 * 4-bit radix pass inside the threshold bin).  ws : csa_workspace_size(CSA_OP_TOPK_BF16, cfg,
 * rows, n_cols) bytes (0 except for few long rows).
 */
csa_status csa_topk_bf16(const csa_config *cfg, const void *scores, int64_t ld, int64_t rows, int64_t n_cols,
                         const int32_t *n_valid, const int32_t *cand, int32_t *idx, void *ws, size_t ws_bytes,
                         csa_stream_t stream);

/*
 * csa_topk_noalloc — csa_topk for callers that cannot allocate device memory.  There is no
 * counterpart in the source pages; it exists for callers that are only ever given input and
 * output buffers (for example a plugin inside another runtime that owns all device memory,
 * or a latency-critical path where an allocation could block or fail), so they cannot pass
 * csa_topk a workspace.
 *
 * Same arguments and results as csa_topk, without ws/ws_bytes.  The scratch is a fixed array
 * of CSA_NOALLOC_SCRATCH_BYTES inside the library (a __device__ object that every GPU which
 * loads the library holds until the process exits); this call allocates nothing.  Sizes whose
 * scratch need (csa_workspace_size(CSA_OP_TOPK, ...)) exceeds that limit are rejected with
 * CSA_ERR_WORKSPACE before anything is launched.
 *  - The first call in a CUDA context (with that context's device current) looks up the
 *    array's device address with cudaGetSymbolAddress, and a call looks it up again when the
 *    current context has changed since (after a device reset, for example); make the first
 *    call in a context before any stream capture.
 *  - All calls share the one array and find it as the previous call left it; what must start
 *    at zero is cleared on the stream.  Calls whose work overlaps on the GPU (different streams,
 *    or different host threads without ordering) race on it: order them on one stream.
 */
#define CSA_NOALLOC_SCRATCH_BYTES (4u << 20)
csa_status csa_topk_noalloc(const csa_config *cfg, const float *scores, int64_t ld, int64_t rows,
                            int64_t n_cols, const int32_t *n_valid, const int32_t *cand, int32_t *idx,
                            csa_stream_t stream);

/*
 * csa_block_pool — CSA2 Hierarchical Sparse Indexer candidate pool (V4.1 page, section 3):
 * block j covers positions [block*j, block*(j+1)) ∩ [0, n_valid[r]); its score is the max
 * there; the n_blocks best blocks under (max desc, j asc) are kept and expanded to their
 * visible positions.
 *   pool       : [rows, n_blocks*block] int32, ascending, -1 padded
 *   pool_count : [rows] int32 (number of valid positions), may be NULL
 */
/* Workspace bytes csa_block_pool needs for these sizes ((size_t)-1 if they are invalid). */
size_t csa_block_pool_workspace_size(int64_t rows, int64_t n_cols, int32_t block, int32_t n_blocks);

csa_status csa_block_pool(const csa_config *cfg, const float *scores, int64_t ld, int64_t rows,
                          int64_t n_cols, const int32_t *n_valid, int32_t block, int32_t n_blocks,
                          int32_t *pool, int32_t *pool_count, void *ws, size_t ws_bytes,
                          csa_stream_t stream);

/*
 * csa_sparse_attn — core sparse MQA attention with window and sink ("Key and value are the
 * same vector", "Attention sink, and heads that abstain", "The sliding window is not an
 * optimisation").  For query row r = b*T + t at position p = q_pos[r], the rows are
 *   kv_comp[b, idx[r, j]] for every idx[r, j] >= 0, then
 *   kv_local[b, p' - local_base[b]] for p' in [max(0, p-W+1), p] ∩ [local_base, local_base+L)
 * each used as both key and value; per head h with l_j = softmax_scale * q[r,h] . row_j:
 *   out[r, h] = sum_j e^{l_j} row_j / (sum_j e^{l_j} + e^{sink[h]}),
 *   lse[r, h] = log(sum_j e^{l_j} + e^{sink[h]}).
 *
 *   q : [B, T, H, d]; kv_comp : [B, E_cap, d]; idx : [B*T, k] int32 (-1 = empty slot;
 *   >= E_cap is skipped and reported as CSA_ERR_INDEX); kv_local : [B, L, d];
 *   local_base, q_pos : int64 [B] and [B*T]; sink : [H] fp32; out : [B, T, H, d] (cfg->act);
 *   lse : [B, T, H] fp32 or NULL.
 * bf16 with d == 512, H == 64 runs on the tcgen05 tensor cores; other shapes with d <= 128,
 * H <= 64 run a CUDA-core path.
 */
csa_status csa_sparse_attn(const csa_config *cfg, const void *q, int32_t T, const void *kv_comp,
                           int64_t E_cap, const int32_t *idx, const void *kv_local, int64_t L,
                           const int64_t *local_base, const int64_t *q_pos, const float *sink,
                           void *out, float *lse, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_dense_attn — HCA core attention ("Heavily Compressed Attention": no indexer and no
 * top-k, the layer attends to every entry it holds; window and per-head sink as in
 * csa_sparse_attn).  For query row r = b*T + t at position p = q_pos[r] the rows are
 *   kv_comp[b, s] for s < min(floor((p+1)/cfg->m), E_cap), then the window rows of
 *   csa_sparse_attn; out and lse as there.
 * Only cfg->B, H, d, m, W, act and softmax_scale are read.
 *   ws : csa_workspace_size(CSA_OP_DENSE_ATTN, cfg, B*T, E_cap) bytes (0 when many queries
 *        share the launch; few queries split their rows over CTAs and merge partials in ws)
 * bf16 with d == 512, H == 64 runs on the tcgen05 tensor cores; other shapes with d <= 128,
 * H <= 64 run a CUDA-core path.
 */
csa_status csa_dense_attn(const csa_config *cfg, const void *q, int32_t T, const void *kv_comp,
                          int64_t E_cap, const void *kv_local, int64_t L, const int64_t *local_base,
                          const int64_t *q_pos, const float *sink, void *out, float *lse, void *ws,
                          size_t ws_bytes, csa_stream_t stream);

/* All inputs of one HCA decode token per sequence (T = 1). */
typedef struct {
  int64_t E_cap;             /* rows of kv_comp per sequence                                   */
  const int64_t *q_pos;      /* [B] position t of the new token                                */
  const void *q;             /* [B, H, d]                                                      */
  const float *sink;         /* [H]                                                            */
  void *kv_comp;             /* [B, E_cap, d]  row (t+1)/m - 1 written when (t+1) % m == 0     */
  const void *kv_tail;       /* [B, m, d]  C of tokens t-m+1 .. t                              */
  const void *z_tail;        /* [B, m, d]  Z of the same tokens                                */
  const float *bias;         /* [m, d] fp32 or NULL                                            */
  const void *kv_local;      /* [B, L, d] uncompressed window rows                             */
  int64_t L;
  const int64_t *local_base; /* [B] position of kv_local[b, 0]                                 */
  void *out;                 /* [B, H, d]                                                      */
  float *lse;                /* [B, H] or NULL                                                 */
} csa_hca_decode_args;

/*
 * csa_hca_decode_step — one HCA decode token per sequence: compress the block the token
 * completes (only when (t+1) % m == 0; m = cfg->m, e.g. 128) with the one-stream compressor,
 * then attend densely over every visible entry plus the window, with the sink.  Same
 * semantics as csa_compress_kv_single followed by csa_dense_attn with T = 1.
 *   ws : csa_workspace_size(CSA_OP_HCA_DECODE, cfg, B, E_cap) bytes
 */
csa_status csa_hca_decode_step(const csa_config *cfg, const csa_hca_decode_args *args, void *ws,
                               size_t ws_bytes, csa_stream_t stream);

/*
 * Attention prologue / epilogue ("Key and value are the same vector": RoPE on exactly the
 * last 64 dims of each head, and RoPE at minus the query position on each head's output;
 * "Grouped output projection": RMSNorm per head on the queries and on the compressed KV
 * entry before core attention).  Conventions of these calls:
 *   RMSNorm   y = x / sqrt(mean over the head's dim of x^2 + eps) * norm_weight[c]
 *   RoPE      on dims [dim - rope_dims, dim): pair (2j, 2j+1) of that slice rotates by angle
 *             pos * rope_theta^(-2j / rope_dims) (x0 cos - x1 sin, x0 sin + x1 cos); the phase
 *             is exact to about 1e-9 rad for any int64 position (64-bit fixed-point turns)
 *   a compressed entry i sits at position m * i (the first token of its block).
 */
typedef struct {
  const float *norm_weight; /* [dim] fp32 RMSNorm weight (16-byte aligned), or NULL: no RMSNorm */
  float eps;                /* RMSNorm epsilon, e.g. 1e-6                                        */
  int32_t rope_dims;        /* rotated dims at the end of each head: even, 0 .. min(dim, 128)     */
  float rope_theta;         /* rotary base (> 1), e.g. 10000                                     */
} csa_norm_rope;

/*
 * csa_norm_rope_apply — RMSNorm then RoPE on every (row, head) vector: queries at their
 * positions (q [B*T, H, d], pos = q_pos), window rows (pos = their token positions), or
 * cache entries (pos = m * i).
 *   x, y : [rows, heads, dim] in cfg->act (y may be x); dim % 8 == 0, 8 .. 1024
 *   pos  : [rows] int64
 * Only cfg->act is read (besides B, H, d, m, W checked as in the HCA calls).
 */
csa_status csa_norm_rope_apply(const csa_config *cfg, const void *x, void *y, int64_t rows, int32_t heads,
                               int32_t dim, const int64_t *pos, const csa_norm_rope *nr,
                               csa_stream_t stream);

/*
 * csa_compress_kv_norm_rope — the compressor fused with RMSNorm, RoPE at the entry's
 * position m * i, and the store into the cache (the fusion vLLM applies to the compressor):
 *   streams = 2: the gated two-stream compressor of csa_compress_kv (kv, z [B, n_tok, 2, dim],
 *                bias [2, m, dim] required; entry i needs tokens m(i-1) .. m(i+1)-1);
 *   streams = 1: the one-stream compressor of csa_compress_kv_single (kv, z [B, n_tok, dim],
 *                bias [m, dim] or NULL).
 *   dim % 64 == 0, 64 .. 1024; out [B, E_cap, dim] in cfg->act; rows outside
 *   [ent_begin, ent_end) untouched.  m = cfg->m.
 */
csa_status csa_compress_kv_norm_rope(const csa_config *cfg, int32_t streams, int32_t dim, const void *kv,
                                     const void *z, const float *bias, int64_t n_tok, int64_t tok0,
                                     int64_t ent_begin, int64_t ent_end, void *out, int64_t E_cap,
                                     const csa_norm_rope *nr, csa_stream_t stream);

/*
 * csa_inverse_rope_quant — RoPE at position -pos[r] on the last rope_dims dims of every head
 * of the attention output o [rows, cfg->H, cfg->d] (cfg->act), written to out as cfg->act
 * (out may be o), or, with out_dtype CSA_E4M3, as e4m3 codes [rows, H, d] with one fp32 scale
 * per (row, head) in out_scale [rows, H]: scale = amax/448 of the rotated vector (1 for an
 * all-zero vector), code = e4m3_rn_satfinite(x / scale).  cfg->d % 8 == 0, <= 1024;
 * rope_dims even, <= min(cfg->d, 128).
 */
csa_status csa_inverse_rope_quant(const csa_config *cfg, const void *o, int64_t rows, const int64_t *pos,
                                  int32_t rope_dims, float rope_theta, void *out, csa_dtype out_dtype,
                                  float *out_scale, csa_stream_t stream);

/*
 * FP8 main-KV entries ("What the cache costs, checked four ways": the 64 RoPE dims in bf16 and
 * the other 448 in FP8, 576 bytes an entry): bytes [0, d-64) are e4m3 codes of dims 0 .. d-65
 * (round to nearest even, saturating at +-448, no scale: RMSNorm keeps the entries well inside
 * that range), bytes [d-64, d+64) the last 64 dims in bf16 (little endian).
 *
 * csa_kv_pack_fp8 — rows x [rows, dim] (cfg->act) -> out [rows, dim + 64] bytes; dim % 16 == 0,
 *                   64 < dim <= 1024.
 * csa_compress_kv_norm_rope_fp8kv — csa_compress_kv_norm_rope writing FP8 entries:
 *                   out [B, E_cap, dim + 64] bytes.
 * csa_sparse_attn_fp8kv — csa_sparse_attn with kv_comp [B, E_cap, 576] FP8 entries (the rows
 *                   are widened to bf16 in shared memory before the tensor-core products, exactly,
 *                   so the result equals csa_sparse_attn over the decoded cache); window rows
 *                   stay cfg->act.  bf16, H = 64, d = 512, and either few queries (B*T below the
 *                   SM count, k + W > 128: the decode split plan) or one CTA a query (many
 *                   queries, such as a prefill chunk; k <= 2048); CSA_ERR_SHAPE otherwise.
 *                   Workspace: csa_workspace_size(CSA_OP_ATTN, ...).
 */
csa_status csa_kv_pack_fp8(const csa_config *cfg, const void *x, int64_t rows, int32_t dim, void *out,
                           csa_stream_t stream);
csa_status csa_compress_kv_norm_rope_fp8kv(const csa_config *cfg, int32_t streams, int32_t dim,
                                           const void *kv, const void *z, const float *bias, int64_t n_tok,
                                           int64_t tok0, int64_t ent_begin, int64_t ent_end, void *out,
                                           int64_t E_cap, const csa_norm_rope *nr, csa_stream_t stream);
csa_status csa_sparse_attn_fp8kv(const csa_config *cfg, const void *q, int32_t T, const void *kv_comp,
                                 int64_t E_cap, const int32_t *idx, const void *kv_local, int64_t L,
                                 const int64_t *local_base, const int64_t *q_pos, const float *sink,
                                 void *out, float *lse, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * MXFP4 main-KV entries (V4.1 page, section 4: E2M1 payloads with one E4M3 scale per 16
 * channels, no global scale; 288 bytes for 512 channels): per block of 16 channels the scale
 * is e4m3_rn_satfinite(amax / 6) and each code the nearest E2M1 value (0, 0.5, 1, 1.5, 2, 3, 4,
 * 6; ties to the even code, saturating, sign kept) of x / scale, both quotients in binary32
 * (a zero scale gives zero codes); element 2i sits in the low nibble of payload byte i; bytes
 * [0, d/2) are the payload, [d/2, d/2 + d/16) the scales.
 *
 * csa_kv_pack_mxfp4 — rows x [rows, dim] (cfg->act) -> out [rows, dim/2 + dim/16] bytes;
 *                     dim % 128 == 0, <= 1024.
 * csa_sparse_attn_mxfp4kv — csa_sparse_attn_fp8kv over MXFP4 entries (kv_comp [B, E_cap, 288]):
 *                     the same shapes, widened to bf16 in shared memory (exactly).
 */
csa_status csa_kv_pack_mxfp4(const csa_config *cfg, const void *x, int64_t rows, int32_t dim, void *out,
                             csa_stream_t stream);
csa_status csa_sparse_attn_mxfp4kv(const csa_config *cfg, const void *q, int32_t T, const void *kv_comp,
                                   int64_t E_cap, const int32_t *idx, const void *kv_local, int64_t L,
                                   const int64_t *local_base, const int64_t *q_pos, const float *sink,
                                   void *out, float *lse, void *ws, size_t ws_bytes, csa_stream_t stream);

/* All inputs of one decode token per sequence (T = 1). */
typedef struct {
  int64_t E_cap;             /* rows of kv_comp / kI / kscale per sequence                    */
  const int64_t *q_pos;      /* [B] position t of the new token                               */
  const void *q;             /* [B, H, d]                                                     */
  const void *qI;            /* [B, HI, dI]                                                   */
  const float *w;            /* [B, HI]                                                       */
  const float *sink;         /* [H]                                                           */
  void *kv_comp;             /* [B, E_cap, d]    row (t+1)/m - 1 rewritten when (t+1) % m == 0 */
  void *kI;                  /* [B, E_cap, dI]   (cfg->kidx; MXFP4: [B, E_cap, 64]), same row  */
  void *kscale;              /* [B, E_cap] fp32 (CSA_E4M3) or scale words (CSA_MXFP4)         */
  const void *kv_tail;       /* [B, 2m, 2, d]  C^a/C^b of tokens t-2m+1 .. t                  */
  const void *z_tail;        /* [B, 2m, 2, d]  Z^a/Z^b of the same tokens                     */
  const void *kvI_tail;      /* [B, 2m, 2, dI] indexer-key streams of the same tokens          */
  const void *zI_tail;       /* [B, 2m, 2, dI]                                                */
  const float *bias;         /* [2, m, d]                                                     */
  const float *biasI;        /* [2, m, dI]                                                    */
  const void *kv_local;      /* [B, L, d] uncompressed window rows                            */
  int64_t L;
  const int64_t *local_base; /* [B] position of kv_local[b, 0]                                */
  void *out;                 /* [B, H, d]                                                     */
  float *lse;                /* [B, H] or NULL                                                */
  int32_t *idx_out;          /* [B, k] or NULL: the entries the step selected                 */
  float *scores_out;         /* [B, E_cap] fp32 (BF16 with bf16_scores) or NULL: the indexer
                                scores the step selected from (-inf past the visible entries);
                                NULL keeps them in ws                                          */
  int32_t bf16_scores;       /* non-zero: the scores are rounded to BF16 (nearest even) before
                                the selection, which then runs on them ("FP4, down to the index
                                scores": BF16 index scores for the selector)                   */
} csa_decode_args;

/*
 * csa_decode_step — one decode token per sequence: compress the block the token completes
 * (only when (t+1) % m == 0), score the visible entries with the lightning indexer, keep the
 * top-k, and attend over them plus the window with the sink.  Same semantics as calling
 * csa_compress_kv (main KV and indexer keys), csa_indexer_scores, csa_topk and
 * csa_sparse_attn in that order with T = 1.
 *
 * Workspace state: the first bytes of ws (a fixed size that depends on cfg->B only) carry
 * the top-k histograms and step counters a sequence from one step to the next (the attention
 * starts on a sequence as soon as its selection's candidates, then its threshold, are
 * counted ready).  ws must be
 * zeroed before the first call (csa_decode_step_reset, or a zero-filled allocation), every
 * call leaves that region ready for the next (also when a bounded wait gives up), and it must
 * not be handed to other calls in between.  Steps on one ws must run in stream order.
 */
csa_status csa_decode_step(const csa_config *cfg, const csa_decode_args *args, void *ws,
                           size_t ws_bytes, csa_stream_t stream);

/*
 * csa_decode_step_reset — zero the part of a decode-step workspace that carries state from
 * one step to the next: its first 4 * 4166 * cfg->B bytes (per sequence a 4096-bin top-k
 * histogram with its ticket, three step counters and the selection's published threshold),
 * asynchronously on `stream`.  Only cfg->B is read.  A step leaves that state ready for the
 * next (histograms and tickets zero, the counters consistent) even when its bounded waits give
 * up (CSA_ERR_TIMEOUT); call this
 * before the first step on a workspace that was not zero-filled, and after a step whose
 * launches failed (CSA_ERR_CUDA) or were never run.
 * Errors: CSA_ERR_NULL (cfg or ws NULL), CSA_ERR_SHAPE (cfg->B < 1), CSA_ERR_ALIGN (ws not
 * 16-byte aligned), CSA_ERR_WORKSPACE (ws_bytes below that size), CSA_ERR_CUDA (the memset
 * could not be enqueued).  Nothing is written on an error.
 */
csa_status csa_decode_step_reset(const csa_config *cfg, void *ws, size_t ws_bytes, csa_stream_t stream);

/*
 * csa_decode_step_fp8kv — csa_decode_step over a main-KV cache of FP8 entries (kv_comp
 * [B, E_cap, 576] bytes, the format of csa_kv_pack_fp8): the entry the token completes is
 * written as an FP8 entry and the attention reads FP8 entries.  bf16, d == 512, m <= 8, the
 * tensor-core indexer and the decode split plan (see csa_sparse_attn_fp8kv); CSA_ERR_SHAPE
 * otherwise.  Same workspace as csa_decode_step.
 */
csa_status csa_decode_step_fp8kv(const csa_config *cfg, const csa_decode_args *args, void *ws,
                                 size_t ws_bytes, csa_stream_t stream);

/*
 * csa_decode_step_mxfp4kv — csa_decode_step over a main-KV cache of MXFP4 entries (kv_comp
 * [B, E_cap, 288] bytes, the format of csa_kv_pack_mxfp4: V4.1 section 4 "FP4: the norm
 * argument…"): the entry the token completes is written as an MXFP4 entry (per 16 channels
 * scale = e4m3(amax / 6), codes = nearest E2M1 value of x / scale) and the attention reads
 * MXFP4 entries.  Same shapes, limits and workspace as csa_decode_step_fp8kv.
 */
csa_status csa_decode_step_mxfp4kv(const csa_config *cfg, const csa_decode_args *args, void *ws,
                                   size_t ws_bytes, csa_stream_t stream);

/* Synchronise `stream`, then return and clear the first device-side error recorded since the
 * last call (CSA_OK if none; CSA_ERR_CUDA if the stream itself reports an error). */
csa_status csa_get_last_error(csa_stream_t stream);

/* Static description of a status code. */
const char *csa_status_string(csa_status s);

/* Number of kernels this process has enqueued through libcsa so far (all devices). */
int64_t csa_launch_count(void);

/*
 * csa_debug_set — fault-injection hooks for tests of the failure path; the pages have no
 * counterpart.  Process-wide; they apply to the csa_decode_step / csa_decode_step_fp8kv calls
 * made after them (the indexer launch of the step):
 *   CSA_DEBUG_WAIT_BUDGET_NS : budget of the launch's bounded device waits, 1e3 .. 2e9 ns
 *                              (default 2e9); CSA_ERR_SHAPE outside that range.
 *   CSA_DEBUG_SKIP_KEY_LOADS : nonzero makes the indexer's producer issue no key-tile load, so
 *                              its consumers' waits run out: the step records CSA_ERR_TIMEOUT
 *                              (read with csa_get_last_error), every kernel role still reaches
 *                              its exit, the step's selection is empty and the workspace state
 *                              is left clean for the next step.  0 (default) turns it off.
 * Leave both at their defaults outside such tests.
 */
typedef enum { CSA_DEBUG_WAIT_BUDGET_NS = 0, CSA_DEBUG_SKIP_KEY_LOADS = 1 } csa_debug_knob;
csa_status csa_debug_set(csa_debug_knob knob, int64_t value);

/* Library version, major*10000 + minor*100 + patch. */
int32_t csa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H_ */
