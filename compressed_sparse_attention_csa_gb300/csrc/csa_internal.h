// Internal launch interface between the C ABI (csa_api.cu) and the kernel translation units.
#pragma once
#include <cstddef>
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "csa.h"

namespace csa {

// Budget of a device-side bounded wait, after which it records CSA_ERR_TIMEOUT and gives up.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// Unique id of the CUDA context current on this thread (0 when none is current or the driver
// cannot tell).  Device addresses of the library's __device__ objects and kernel attributes
// belong to a context, so caches of them are keyed by this id (a device reset or a new
// primary context gets a new id).
unsigned long long current_context_id();
// True the first time the call site owning `slot` runs in the current context (and whenever
// the context cannot be identified): the site then sets its kernels' attributes, which are
// per context.  Thread-safe; setting an attribute twice is harmless.
bool first_use_in_context(std::atomic<unsigned long long>& slot);

// ---- compression ------------------------------------------------------------------
struct CompressJob {    // one cache produced by the compressor
  const void* kv;       // [B, n_tok, 2, dim]
  const void* z;        // [B, n_tok, 2, dim]
  const float* bias;    // [2, m, dim]
  int dim;              // <= 512
  void* out;            // [B, E_cap, dim] (MXFP4: [B, E_cap, dim/2] payload bytes)
  int out_dtype;        // CSA_F32 / CSA_BF16 / CSA_E4M3 / CSA_MXFP4 (dim 128)
  void* out_scale;      // [B, E_cap]: fp32 scales (e4m3) or UE8M0 scale words (MXFP4)
};
struct CompressArgs {
  CompressJob job[2];
  int n_jobs;
  int B, m;             // m <= 16
  bool act_bf16;        // input dtype
  int64_t n_tok, tok0;  // uniform mode: stream row r holds token tok0 + r
  int64_t ent_begin, n_ent;
  const int64_t* q_pos; // decode mode (non-null): per sequence t = q_pos[b]; rows hold t-2m+1..t;
                        // the entry (t+1)/m - 1 is produced only when (t+1) % m == 0
  int64_t E_cap;
  int* err;
  uint32_t* zero_hist;  // decode step: per-sequence top-k histogram rows [B, 4096] and the B
                        // candidate counters after them, zeroed here before the indexer runs
  // decode step: the indexer's query images are prepared in the same launch (extra CTAs
  // along z after the compression jobs); qp_ctas = 0 disables it
  int qp_ctas;
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);

// One-stream compression without overlap (HCA at m' = 128, the CSA2 encoder at m = 2):
// entry i = per-channel softmax over the m logits Z[m i + j] (+ bias[j]) of its own block,
// weighted sum of C over the same tokens.
struct Compress1Args {
  const void* kv;         // [B, n_tok, dim]: C of tokens tok0 .. (decode: [B, m, dim], t-m+1 .. t)
  const void* z;          // same layout: gate logits Z
  const float* bias;      // [m, dim] or null (no positional bias)
  void* out;              // [B, E_cap, dim] (act dtype)
  int B, m, dim;          // dim even
  bool act_bf16;          // stream and output dtype: bf16 (else fp32)
  int64_t n_tok, tok0;    // uniform mode: stream row r holds token tok0 + r
  int64_t ent_begin, n_ent;
  const int64_t* q_pos;   // decode mode (non-null): entry (t+1)/m - 1 when (t+1) % m == 0
  int64_t E_cap;
};
cudaError_t launch_compress1(const Compress1Args& a, cudaStream_t s);

// ---- indexer ----------------------------------------------------------------------
// Decode step (T = 1, tensor-core path): the indexer launch also compresses the entry the
// new token completes (main KV spread over the CTAs of each sequence, indexer key by the CTA
// that scores it, before that tile is loaded), builds its query image in shared memory, and
// histograms its scores into `hist` ([B][4160] rows), which the top-k kernel reads and
// leaves zero again: zero before the first step.
struct DecodeFuse {
  bool on;
  const void* kv_tail;   // [B, 2m, 2, d] tokens t-2m+1..t (stream a, stream b)
  const void* z_tail;
  const float* bias;     // [2, m, d]
  void* kv_comp;         // [B, E_cap, d]
  int d;
  const void* kvI_tail;  // [B, 2m, 2, dI]
  const void* zI_tail;
  const float* biasI;    // [2, m, dI]
  bool act_bf16;         // stream and kv_comp dtype
  int kv_fmt;            // kv_comp rows: 0 the activation dtype; 1 FP8 main-KV entries (d - 64 e4m3
                         // codes, then 64 bf16 dims); 2 MXFP4 entries (d/2 E2M1 bytes, d/16 e4m3 scales)
  uint32_t* hist;        // histograms
};
// decode-step state kept across steps: the histograms [B][4160], the top-k tickets [B] (zero
// before the first step, left zero by every step), then two step counters [B] each: selections
// completed (the selection's last CTA of a row adds one) and selections consumed (the split
// merge copies the first after the step's attention), zero before the first step and left
// equal; the chunks' counters [B] (left zero by the merge) and the published thresholds [B][2]
inline size_t decode_state_words(int B) { return static_cast<size_t>(B) * 4160 + 6 * static_cast<size_t>(B); }
struct IndexerArgs {
  const void* qI;        // [B*T, HI, dI]
  const float* w;        // [B*T, HI]
  const int64_t* q_pos;  // [B*T]
  const void* kI;        // [B, E_cap, dI] (MXFP4: [B, E_cap, 64] payload bytes)
  const void* kscale;    // [B, E_cap]: fp32 scales (e4m3) or UE8M0 scale words (MXFP4)
  const int32_t* cand;   // [B*T, n_cand] or null
  int n_cand;
  float* scores;         // [B*T, ld] fp32, or BF16 when scores_bf16
  int64_t ld;
  int B, T, HI, dI, m;
  int64_t E_cap;
  int act;               // CSA_F32 / CSA_BF16
  int kidx;              // CSA_F32 / CSA_BF16 / CSA_E4M3 / CSA_MXFP4
  int* err;
  int num_sms;
  int32_t* nv_out;       // [B*T] visible-entry count per query row, or null
  uint32_t* hist_out;    // [B*T, 4160] digit histogram of the visible scores (one query per CTA
                         // only), accumulated with atomics; null = none
  void* ws;              // tensor-core path: query images (indexer_workspace_bytes)
  bool images_ready;     // the query images in ws were already written (fused decode prep)
  DecodeFuse fuse;       // decode step only
  bool scores_bf16 = false;           // write the scores rounded to BF16 (RNE), 2 bytes each
  uint64_t wait_ns = kDefaultWaitNs;  // budget of every bounded wait of the launch
  bool skip_key_loads = false;        // fault injection (tests): the producer issues no key load
};
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s);
bool indexer_uses_tensor_cores(const IndexerArgs& a);
size_t indexer_workspace_bytes(const IndexerArgs& a);

// Tensor-core indexer plan (see k_indexer.cu).
struct IndexerLayout {
  int G;               // queries per CTA
  int N;               // MMA N = G * HI
  int stages;
  uint32_t b_bytes;    // B operand image (bf16 rows, or e4m3 hi + lo regions), 1024-aligned
  uint32_t w_bytes;    // gate vector image (G*HI fp32), 16-aligned
  uint32_t stage_bytes;
  uint32_t smem_bytes;
  uint32_t tmem_cols;
  int n_acc;           // TMEM accumulators in the MMA -> epilogue ring (2..4)
  int n_splits;        // key-range splits per (sequence, query group)
  int n_qgroups;
  bool wide;           // one CTA per SM (many query groups); else two, with the key range split
};
IndexerLayout indexer_layout(const IndexerArgs& a);

// The compressor launch of the decode step also writes the indexer's query images: the
// arguments of that part (set by the caller with qp_ctas > 0 in CompressArgs).
struct QprepPart {
  IndexerArgs ia;
  IndexerLayout L;
  uint8_t* images;
  bool fp8;
};
cudaError_t launch_compress_with_qprep(const CompressArgs& a, const QprepPart& q, cudaStream_t s);

// ---- top-k ------------------------------------------------------------------------
struct TopkArgs {
  const void* scores;    // [rows, ld] fp32, or BF16 (bf16 = true)
  int64_t ld, rows, n_cols;
  const int32_t* n_valid;
  const int32_t* cand;   // [rows, n_cols] or null
  int k;
  int32_t* idx;          // [rows, k]
  void* ws;
  size_t ws_bytes;
  int* err;
  int num_sms;
  bool bf16 = false;     // BF16 scores: the histogram and row paths only
};
size_t topk_workspace_bytes(int64_t rows, int64_t n_cols, int k, int num_sms, bool bf16 = false);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);

// Histogram-guided top-k for a few long rows.  hist_cnt holds, per row, 4096 fine digit
// counts (key >> 20) and 64 coarse counts (key >> 26), then one ticket word per row; all
// zero before the histogram is filled.
constexpr int kTopkHistBins = 4096;
constexpr int kTopkHistCoarse = 64;
constexpr int kTopkHistRowWords = kTopkHistBins + kTopkHistCoarse;
int topk_hist_cap(int k);
size_t topk_hist_workspace_bytes(int64_t rows, int64_t n_cols);  // the candidate slots (ws_cand)
bool topk_uses_hist(int64_t rows, int64_t n_cols, bool has_cand);
// Many long rows: one CTA per row with a shared-memory histogram (no workspace).
bool topk_uses_rows(int64_t rows, int64_t n_cols, bool has_cand, int k);
cudaError_t launch_topk_rows(const void* scores, int64_t ld, int64_t rows, int64_t n_cols, const int32_t* n_valid,
                             int k, int32_t* idx, cudaStream_t s, const int32_t* cmap = nullptr, bool bf16 = false);
size_t topk_hist_standalone_bytes(int64_t rows, int64_t n_cols);
cudaError_t launch_topk_hist_standalone(const TopkArgs& a, cudaStream_t s);
// hist_cnt: [rows][4160] then rows tickets; left zero for the next use.
// Decode-step extras of the histogram selection (all null / zero: none).
struct SelHandoff {
  uint32_t* done;            // [rows] counters the row's last CTA increments once its list is written
                             // (or, with cand_cap, once its threshold is published)
  uint32_t* chunks;          // [rows] counters every chunk CTA increments once its slot is written
  uint32_t* thr;             // [rows][2]: threshold key T and tie cut P of the published threshold
  int cand_cap;              // > 0: rows with at most cand_cap candidates publish (T, P) and count
                             // done before writing the list (a candidate wins iff key > T, or
                             // key == T and position <= P); others count done after the list
  const uint8_t* pf_rows;    // cache rows the list indexes: every candidate's row (row r's entry s at
  int64_t pf_row_bytes;      // pf_rows + (r * pf_seq_rows + s) * pf_row_bytes, a multiple of 16
  int64_t pf_seq_rows;       // bytes) is prefetched into L2 as soon as its chunk keeps it
};
// The selection's per-chunk candidate slots in the top-k workspace (ws_cand of launch_topk_hist):
// row r's chunk c at words ((r * n_chunks + c) * sel_slot_words(); [count, 3 pad][keys x
// sel_slot_cap()][positions x sel_slot_cap()]; n_chunks = sel_chunks(n_cols).
int sel_slot_words();
int sel_slot_cap();
int sel_chunks(int64_t n_cols);
cudaError_t launch_topk_hist(const void* scores, int64_t ld, int64_t rows, int64_t n_cols, const int32_t* n_valid,
                             uint32_t* hist_cnt, int k, int32_t* idx, void* ws_cand, int num_sms, cudaStream_t s,
                             const int32_t* cmap = nullptr, bool bf16 = false, const SelHandoff& ho = SelHandoff{});

struct PoolArgs {
  const float* scores;
  int64_t ld, rows, n_cols;
  const int32_t* n_valid;
  int block, n_blocks;
  int32_t* pool;         // [rows, n_blocks*block]
  int32_t* pool_count;   // [rows] or null
  void* ws;
  size_t ws_bytes;
  int* err;
  int num_sms;
};
size_t pool_workspace_bytes(int64_t rows, int64_t n_cols, int block, int n_blocks, int num_sms);
cudaError_t launch_block_pool(const PoolArgs& a, cudaStream_t s);

// ---- attention --------------------------------------------------------------------
struct AttnArgs {
  const void* q;          // [B*T, H, d]
  const void* kv_comp;    // [B, E_cap, d]
  const int32_t* idx;     // [B*T, k]
  const void* kv_local;   // [B, L, d]
  const int64_t* local_base;
  const int64_t* q_pos;
  const float* sink;      // [H]
  void* out;              // [B*T, H, d]
  float* lse;             // [B*T, H] or null
  int B, T, H, d, k, W;
  int64_t E_cap, L;
  float softmax_scale;
  int act;
  int dense_m;            // > 0: no idx; the entries are every s < min(floor((t+1)/dense_m), E_cap)
  int dense_step;         // dense decode step: the kernel before is the step's compressor (it
                          // writes only entry floor((t+1)/dense_m) - 1, after its own wait)
  uint32_t* sel_done;     // sparse decode step (or null): [B] selections completed, counted by the
  uint32_t* sel_seen;     // selection kernel before this one; [B] selections consumed (the merge
                          // sets it to sel_done): query r's list is ready once sel_done[r] passes
                          // sel_seen[r], and holds its entries first (ascending), then -1
  int cand_cap;           // > 0 (with sel_done): candidate mode for rows of at most cand_cap
                          // candidates (see SelHandoff): split 0 the window, split s > 0 the
                          // candidates 128 (s - 1) .. +127, masked by the published threshold
  uint32_t* sel_chunks;   // [B] chunk counters (the merge zeroes them after the step)
  const uint32_t* sel_thr;    // [B][2] published thresholds
  const uint32_t* sel_slots;  // the selection's candidate slots
  int sel_n_chunks, sel_slot_words, sel_slot_cap;
  int min_split;          // decode split plan: at least this many splits
  void* ws;
  size_t ws_bytes;
  int* err;
  int num_sms;
};
size_t attn_workspace_bytes(int B, int T, int H, int d, int k, int W, int act, int num_sms, int min_split = 0);
// Dense (HCA) attention: workspace for the split plan over at most E_cap + W rows a query.
size_t attn_dense_workspace_bytes(int B, int T, int H, int d, int64_t E_cap, int W, int act, int num_sms);
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s);

// ---- shared host utilities ---------------------------------------------------------
int device_sm_count();
void count_launches(int n);  // bookkeeping for csa_launch_count()
bool encode_tmap_generic(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch with programmatic stream serialization (the kernel must call pdl_wait() before it
// reads what earlier kernels on the stream wrote).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace csa
