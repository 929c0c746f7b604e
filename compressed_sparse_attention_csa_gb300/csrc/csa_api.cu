// C ABI of libcsa: argument validation, workspace planning, the device error word, TMA
// descriptor encoding and the fused decode step.  Every entry point validates on the host,
// then enqueues kernels on the caller's stream; nothing here allocates memory.
#include <cmath>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "csa_internal.h"
#include "csa_epi.h"

namespace csa {

// ------------------------------------------------------------------ device state
static __device__ int g_err_word;  // first device-side error since the last read

static constexpr int kMaxDevices = 64;

unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

bool first_use_in_context(std::atomic<unsigned long long>& slot) {
  const unsigned long long id = current_context_id();
  if (id == 0) return true;
  return slot.exchange(id) != id;
}

// Device address of g_err_word in the current context (looked up again when the context
// changes).
static int* err_word_ptr() {
  struct Slot {
    unsigned long long ctx;
    int* ptr;
  };
  static Slot slots[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!slots[dev].ptr || id == 0 || slots[dev].ctx != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    slots[dev] = Slot{current_context_id(), static_cast<int*>(p)};
  }
  return slots[dev].ptr;
}

static std::atomic<int64_t> g_launches{0};
// fault-injection knobs (csa_debug_set): the decode step's wait budget and skipped key loads
static std::atomic<uint64_t> g_debug_wait_ns{kDefaultWaitNs};
static std::atomic<int> g_debug_skip_loads{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int device_sm_count() {
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;  // planning default when no device is visible (no launch happens then)
  }
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cache[dev] = n;
  }
  return cache[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_tmap_generic(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[5] = {0, 0, 0, 0, 0};
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return fn(map, dtype, static_cast<cuuint32_t>(rank), base, d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace csa

using namespace csa;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The indexer keys of cfg->kidx: scales present for the quantised formats; MXFP4 payloads
// 32-byte aligned (the unpacking TMA's rule) and E_cap a multiple of 4 (a tile's TMA boxes
// take every fourth key of a sequence).
csa_status check_keys(const csa_config* c, const void* kI, const void* kscale, int64_t E_cap) {
  if ((c->kidx == CSA_E4M3 || c->kidx == CSA_MXFP4) && !kscale) return CSA_ERR_NULL;
  if (c->kidx == CSA_MXFP4) {
    if ((reinterpret_cast<uintptr_t>(kI) & 31u) != 0) return CSA_ERR_ALIGN;
    if (E_cap % 4 != 0) return CSA_ERR_SHAPE;
  }
  return CSA_OK;
}

csa_status check_cfg(const csa_config* c) {
  if (!c) return CSA_ERR_NULL;
  if (c->B < 1 || c->H < 1 || c->d < 1 || c->HI < 1 || c->m < 1 || c->k < 1 || c->k > 4096 || c->W < 0)
    return CSA_ERR_SHAPE;
  if (c->dI != 32 && c->dI != 64 && c->dI != 128) return CSA_ERR_SHAPE;
  if (c->act != CSA_F32 && c->act != CSA_BF16) return CSA_ERR_DTYPE;
  if (c->kidx != c->act && c->kidx != CSA_E4M3 && c->kidx != CSA_MXFP4) return CSA_ERR_DTYPE;
  if (c->kidx == CSA_MXFP4 && c->act != CSA_BF16) return CSA_ERR_DTYPE;
  if (c->kidx == CSA_MXFP4 && c->dI != 128) return CSA_ERR_SHAPE;
  if (!std::isfinite(c->softmax_scale)) return CSA_ERR_SHAPE;
  return CSA_OK;
}

csa_status launch_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

// The calls of the HCA path read B, H, d, m, W, act and softmax_scale only.
csa_status check_cfg_hca(const csa_config* c) {
  if (!c) return CSA_ERR_NULL;
  if (c->B < 1 || c->H < 1 || c->d < 1 || c->m < 1 || c->m > 4096 || c->W < 0) return CSA_ERR_SHAPE;
  if (c->act != CSA_F32 && c->act != CSA_BF16) return CSA_ERR_DTYPE;
  if (!std::isfinite(c->softmax_scale)) return CSA_ERR_SHAPE;
  return CSA_OK;
}

bool dense_shape_ok(const csa_config* c) {
  const bool tc = c->act == CSA_BF16 && c->H == 64 && c->d == 512;
  const bool simt = c->d <= 128 && c->H <= 64;
  return tc || simt;
}

bool attn_shape_ok(const csa_config* c) {
  const bool tc = c->act == CSA_BF16 && c->H == 64 && c->d == 512 && c->k <= 2048;
  const bool simt = c->d <= 128 && c->H <= 64;
  return tc || simt;
}

IndexerArgs indexer_shape(const csa_config* c, int T, int64_t E_cap, int sms) {
  IndexerArgs a{};
  a.B = c->B;
  a.T = T;
  a.HI = c->HI;
  a.dI = c->dI;
  a.m = c->m;
  a.E_cap = E_cap;
  a.act = c->act;
  a.kidx = c->kidx;
  a.num_sms = sms;
  return a;
}

// csa_indexer_topk: [query images][scores rows*E_cap*4][visible counts][top-k workspace].
size_t indexer_topk_ws(const csa_config* c, int T, int64_t E_cap, int sms, bool bf16 = false) {
  const int64_t rows = static_cast<int64_t>(c->B) * T;
  return align_up(indexer_workspace_bytes(indexer_shape(c, T, E_cap, sms)), 256) +
         align_up(static_cast<size_t>(rows * E_cap) * (bf16 ? 2 : 4), 256) + align_up(static_cast<size_t>(rows) * 4, 256) +
         align_up(topk_workspace_bytes(rows, E_cap, c->k, sms, bf16), 256);
}

// Candidate mode of the decode step's attention (decode split plan, a window of at most 128
// rows, at most 64 selection chunks, and a grid of 1 + kCandCap / 128 splits a query in at
// least two head groups that still fits the SMs): a row with at most kCandCap candidates is
// attended over its candidates, gathered before the selection's threshold is known and masked
// by it.  (With one head group, B 16 at 64K, the wider grid cost more than the overlap gained.)
constexpr int kCandCap = 1024;
int decode_cand_cap(const csa_config* c, int64_t E_cap, int sms) {
  if (!attn_fp8kv_supported(c->B, 1, c->H, c->d, c->k, c->W, c->act, sms)) return 0;
  if (c->W > 128 || sel_chunks(E_cap) > 64 || kCandCap > sel_slot_cap()) return 0;
  if (static_cast<int64_t>(1 + kCandCap / 128) * c->B * 2 > sms) return 0;
  return kCandCap;
}

size_t decode_ws(const csa_config* c, int64_t E_cap, int sms) {
  const int64_t B = c->B;
  // first, at a fixed offset: the top-k histograms and tickets kept across steps
  size_t bytes = align_up(decode_state_words(static_cast<int>(B)) * 4, 256);
  bytes += align_up(indexer_workspace_bytes(indexer_shape(c, 1, E_cap, sms)), 256);  // query images
  bytes += align_up(static_cast<size_t>(B * E_cap) * 4, 256);  // scores
  bytes += align_up(static_cast<size_t>(B) * 4, 256);                 // visible counts
  bytes += align_up(static_cast<size_t>(B) * c->k * 4, 256);          // idx
  bytes += align_up(std::max(topk_workspace_bytes(B, E_cap, c->k, sms), topk_hist_workspace_bytes(B, E_cap)), 256);
  const int cap = decode_cand_cap(c, E_cap, sms);
  bytes += align_up(attn_workspace_bytes(c->B, 1, c->H, c->d, c->k, c->W, c->act, sms, cap > 0 ? 1 + cap / 128 : 0), 256);
  return bytes;
}

}  // namespace

extern "C" {

int32_t csa_version(void) { return 100; }

int64_t csa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

csa_status csa_debug_set(csa_debug_knob knob, int64_t value) {
  switch (knob) {
    case CSA_DEBUG_WAIT_BUDGET_NS:
      if (value < 1000 || value > static_cast<int64_t>(kDefaultWaitNs)) return CSA_ERR_SHAPE;
      g_debug_wait_ns.store(static_cast<uint64_t>(value), std::memory_order_relaxed);
      return CSA_OK;
    case CSA_DEBUG_SKIP_KEY_LOADS:
      g_debug_skip_loads.store(value != 0 ? 1 : 0, std::memory_order_relaxed);
      return CSA_OK;
  }
  return CSA_ERR_SHAPE;
}

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_NULL: return "null pointer";
    case CSA_ERR_SHAPE: return "invalid shape";
    case CSA_ERR_DTYPE: return "unsupported dtype";
    case CSA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case CSA_ERR_WORKSPACE: return "workspace too small";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
    case CSA_ERR_INDEX: return "selected index out of range";
  }
  return "unknown status";
}

csa_status csa_get_last_error(csa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return CSA_ERR_CUDA;
  int* p = err_word_ptr();
  if (!p) return CSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CSA_ERR_CUDA;
  }
  return static_cast<csa_status>(v);
}

size_t csa_workspace_size(csa_op op, const csa_config* cfg, int64_t rows, int64_t n_cols) {
  const int sms = device_sm_count();
  if (op == CSA_OP_DENSE_ATTN || op == CSA_OP_HCA_DECODE) {  // rows = B*T (B for the step), n_cols = E_cap
    if (check_cfg_hca(cfg) != CSA_OK || rows < 0 || n_cols < 0 || rows % cfg->B || n_cols > (int64_t(1) << 24) ||
        (op == CSA_OP_HCA_DECODE && rows != cfg->B))
      return static_cast<size_t>(-1);
    return attn_dense_workspace_bytes(cfg->B, static_cast<int>(rows / cfg->B), cfg->H, cfg->d, n_cols, cfg->W,
                                      cfg->act, sms);
  }
  if (check_cfg(cfg) != CSA_OK || rows < 0 || n_cols < 0) return static_cast<size_t>(-1);
  switch (op) {
    case CSA_OP_COMPRESS:
      return 0;
    case CSA_OP_INDEXER: {  // rows = B*T, n_cols = T
      if (n_cols < 1 || rows % n_cols || rows / n_cols != cfg->B) return static_cast<size_t>(-1);
      return indexer_workspace_bytes(indexer_shape(cfg, static_cast<int>(n_cols), 1, sms));
    }
    case CSA_OP_TOPK:
    case CSA_OP_TOPK_BF16:
      if (n_cols > (int64_t(1) << 24)) return static_cast<size_t>(-1);
      return topk_workspace_bytes(rows, n_cols, cfg->k, sms, op == CSA_OP_TOPK_BF16);
    case CSA_OP_ATTN: {
      if (n_cols < 1 || rows % n_cols) return static_cast<size_t>(-1);
      return attn_workspace_bytes(static_cast<int>(rows / n_cols), static_cast<int>(n_cols), cfg->H, cfg->d,
                                  cfg->k, cfg->W, cfg->act, sms);
    }
    case CSA_OP_DECODE:
      if (rows != cfg->B || n_cols > (int64_t(1) << 24)) return static_cast<size_t>(-1);
      return decode_ws(cfg, n_cols, sms);
    case CSA_OP_POOL:
      return static_cast<size_t>(-1);
    case CSA_OP_INDEXER_TOPK:  // rows = B*T, n_cols = E_cap
    case CSA_OP_INDEXER_TOPK_BF16:
      if (rows % cfg->B || n_cols < 1 || n_cols > (int64_t(1) << 24)) return static_cast<size_t>(-1);
      return indexer_topk_ws(cfg, static_cast<int>(rows / cfg->B), n_cols, sms, op == CSA_OP_INDEXER_TOPK_BF16);
    default:
      break;
  }
  return static_cast<size_t>(-1);
}

size_t csa_block_pool_workspace_size(int64_t rows, int64_t n_cols, int32_t block, int32_t n_blocks) {
  if (rows < 0 || n_cols < 0 || block < 1 || n_blocks < 1 || n_blocks > 4096 || n_cols > (int64_t(1) << 24))
    return static_cast<size_t>(-1);
  return pool_workspace_bytes(rows, n_cols, block, n_blocks, device_sm_count());
}

csa_status csa_compress_kv(const csa_config* cfg, int32_t dim, const void* kv, const void* z, const float* bias,
                           int64_t n_tok, int64_t tok0, int64_t ent_begin, int64_t ent_end, void* out,
                           csa_dtype out_dtype, void* out_scale, int64_t E_cap, csa_stream_t stream) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!kv || !z || !bias || !out) return CSA_ERR_NULL;
  if ((out_dtype == CSA_E4M3 || out_dtype == CSA_MXFP4) && !out_scale) return CSA_ERR_NULL;
  if (out_dtype != CSA_F32 && out_dtype != CSA_BF16 && out_dtype != CSA_E4M3 && out_dtype != CSA_MXFP4)
    return CSA_ERR_DTYPE;
  if (out_dtype == CSA_MXFP4 && dim != 128) return CSA_ERR_SHAPE;
  if (!aligned16(kv) || !aligned16(z) || !aligned16(bias) || !aligned16(out) || (out_scale && !aligned16(out_scale)))
    return CSA_ERR_ALIGN;
  if (dim < 1 || dim > 512 || cfg->m > 16 || n_tok < 0 || ent_begin < 0 || ent_end < ent_begin || ent_end > E_cap)
    return CSA_ERR_SHAPE;
  const int64_t m = cfg->m;
  if (ent_end > ent_begin) {
    const int64_t need_lo = ent_begin > 0 ? m * (ent_begin - 1) : 0;
    if (tok0 > need_lo || m * ent_end > tok0 + n_tok) return CSA_ERR_SHAPE;
  }
  CompressArgs a{};
  a.job[0] = CompressJob{kv, z, bias, dim, out, out_dtype, out_scale};
  a.n_jobs = 1;
  a.B = cfg->B;
  a.m = cfg->m;
  a.act_bf16 = cfg->act == CSA_BF16;
  a.n_tok = n_tok;
  a.tok0 = tok0;
  a.ent_begin = ent_begin;
  a.n_ent = ent_end - ent_begin;
  a.E_cap = E_cap;
  a.err = err_word_ptr();
  return launch_status(launch_compress(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_compress_kv_single(const csa_config* cfg, int32_t dim, const void* kv, const void* z,
                                  const float* bias, int64_t n_tok, int64_t tok0, int64_t ent_begin, int64_t ent_end,
                                  void* out, int64_t E_cap, csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!kv || !z || !out) return CSA_ERR_NULL;
  if (!aligned16(kv) || !aligned16(z) || !aligned16(out) || (bias && !aligned16(bias))) return CSA_ERR_ALIGN;
  const int64_t m = cfg->m;
  if (dim < 2 || dim > 4096 || (dim & 1) || n_tok < 0 || ent_begin < 0 || ent_end < ent_begin || ent_end > E_cap ||
      E_cap * cfg->B >= (int64_t(1) << 31))
    return CSA_ERR_SHAPE;
  if (ent_end > ent_begin && (tok0 > m * ent_begin || m * ent_end > tok0 + n_tok)) return CSA_ERR_SHAPE;
  Compress1Args a{};
  a.kv = kv;
  a.z = z;
  a.bias = bias;
  a.out = out;
  a.B = cfg->B;
  a.m = cfg->m;
  a.dim = dim;
  a.act_bf16 = cfg->act == CSA_BF16;
  a.n_tok = n_tok;
  a.tok0 = tok0;
  a.ent_begin = ent_begin;
  a.n_ent = ent_end - ent_begin;
  a.E_cap = E_cap;
  return launch_status(launch_compress1(a, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
csa_status check_norm_rope(const csa_norm_rope* nr, int32_t dim) {
  if (!nr) return CSA_ERR_NULL;
  if (nr->norm_weight && !aligned16(nr->norm_weight)) return CSA_ERR_ALIGN;
  if (nr->rope_dims < 0 || nr->rope_dims > dim || nr->rope_dims > kMaxRopeDims || (nr->rope_dims & 1) ||
      !std::isfinite(nr->eps) || nr->eps < 0.f ||
      (nr->rope_dims > 0 && !(nr->rope_theta > 1.f && std::isfinite(nr->rope_theta))))
    return CSA_ERR_SHAPE;
  return CSA_OK;
}
NormRope to_norm_rope(const csa_norm_rope* nr) {
  NormRope r{};
  r.weight = nr->norm_weight;
  r.eps = nr->eps;
  r.rope_dims = nr->rope_dims;
  r.theta = nr->rope_theta;
  make_rope_table(nr->rope_theta, nr->rope_dims, &r.tab);
  return r;
}
}  // namespace

csa_status csa_norm_rope_apply(const csa_config* cfg, const void* x, void* y, int64_t rows, int32_t heads, int32_t dim,
                               const int64_t* pos, const csa_norm_rope* nr, csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!x || !y || !pos) return CSA_ERR_NULL;
  if (!aligned16(x) || !aligned16(y) || !aligned16(pos)) return CSA_ERR_ALIGN;
  if (rows < 0 || heads < 1 || dim < 8 || dim > 1024 || (dim & 7) || rows * heads >= (int64_t(1) << 40))
    return CSA_ERR_SHAPE;
  st = check_norm_rope(nr, dim);
  if (st != CSA_OK) return st;
  NormRopeArgs a{};
  a.x = x;
  a.y = y;
  a.rows = rows;
  a.heads = heads;
  a.dim = dim;
  a.pos = pos;
  a.bf16 = cfg->act == CSA_BF16;
  a.nr = to_norm_rope(nr);
  return launch_status(launch_norm_rope(a, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
csa_status compress_norm_rope_impl(const csa_config* cfg, int32_t streams, int32_t dim, const void* kv, const void* z,
                                   const float* bias, int64_t n_tok, int64_t tok0, int64_t ent_begin, int64_t ent_end,
                                   void* out, int64_t E_cap, const csa_norm_rope* nr, bool fp8kv, csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!kv || !z || !out || (streams == 2 && !bias)) return CSA_ERR_NULL;
  if (!aligned16(kv) || !aligned16(z) || !aligned16(out) || (bias && !aligned16(bias))) return CSA_ERR_ALIGN;
  const int64_t m = cfg->m;
  if ((streams != 1 && streams != 2) || dim < 64 || dim > 1024 || (dim % 64) || n_tok < 0 || ent_begin < 0 ||
      ent_end < ent_begin || ent_end > E_cap || E_cap * cfg->B >= (int64_t(1) << 31))
    return CSA_ERR_SHAPE;
  if (ent_end > ent_begin) {
    const int64_t need_lo = streams == 2 ? (ent_begin > 0 ? m * (ent_begin - 1) : 0) : m * ent_begin;
    if (tok0 > need_lo || m * ent_end > tok0 + n_tok) return CSA_ERR_SHAPE;
  }
  st = check_norm_rope(nr, dim);
  if (st != CSA_OK) return st;
  CompressEpiArgs a{};
  a.two_stream = streams == 2;
  a.kv = kv;
  a.z = z;
  a.bias = bias;
  a.B = cfg->B;
  a.m = cfg->m;
  a.dim = dim;
  a.n_tok = n_tok;
  a.tok0 = tok0;
  a.ent_begin = ent_begin;
  a.n_ent = ent_end - ent_begin;
  a.E_cap = E_cap;
  a.out = out;
  a.bf16 = cfg->act == CSA_BF16;
  a.fp8kv = fp8kv;
  a.nr = to_norm_rope(nr);
  return launch_status(launch_compress_norm_rope(a, reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace

csa_status csa_compress_kv_norm_rope(const csa_config* cfg, int32_t streams, int32_t dim, const void* kv, const void* z,
                                     const float* bias, int64_t n_tok, int64_t tok0, int64_t ent_begin,
                                     int64_t ent_end, void* out, int64_t E_cap, const csa_norm_rope* nr,
                                     csa_stream_t stream) {
  return compress_norm_rope_impl(cfg, streams, dim, kv, z, bias, n_tok, tok0, ent_begin, ent_end, out, E_cap, nr,
                                 false, stream);
}

csa_status csa_compress_kv_norm_rope_fp8kv(const csa_config* cfg, int32_t streams, int32_t dim, const void* kv,
                                           const void* z, const float* bias, int64_t n_tok, int64_t tok0,
                                           int64_t ent_begin, int64_t ent_end, void* out, int64_t E_cap,
                                           const csa_norm_rope* nr, csa_stream_t stream) {
  return compress_norm_rope_impl(cfg, streams, dim, kv, z, bias, n_tok, tok0, ent_begin, ent_end, out, E_cap, nr,
                                 true, stream);
}

csa_status csa_kv_pack_mxfp4(const csa_config* cfg, const void* x, int64_t rows, int32_t dim, void* out,
                             csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!x || !out) return CSA_ERR_NULL;
  if (!aligned16(x) || !aligned16(out)) return CSA_ERR_ALIGN;
  if (rows < 0 || dim < 16 || dim > 1024 || (dim % 16) || ((dim / 2 + dim / 16) % 8)) return CSA_ERR_SHAPE;
  KvPackArgs a{};
  a.x = x;
  a.out = out;
  a.rows = rows;
  a.dim = dim;
  a.bf16 = cfg->act == CSA_BF16;
  return launch_status(launch_kv_pack_mxfp4(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_kv_pack_fp8(const csa_config* cfg, const void* x, int64_t rows, int32_t dim, void* out,
                           csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!x || !out) return CSA_ERR_NULL;
  if (!aligned16(x) || !aligned16(out)) return CSA_ERR_ALIGN;
  if (rows < 0 || dim <= 64 || dim > 1024 || (dim % 16)) return CSA_ERR_SHAPE;
  KvPackArgs a{};
  a.x = x;
  a.out = out;
  a.rows = rows;
  a.dim = dim;
  a.bf16 = cfg->act == CSA_BF16;
  return launch_status(launch_kv_pack_fp8(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_inverse_rope_quant(const csa_config* cfg, const void* o, int64_t rows, const int64_t* pos,
                                  int32_t rope_dims, float rope_theta, void* out, csa_dtype out_dtype, float* out_scale,
                                  csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!o || !pos || !out || (out_dtype == CSA_E4M3 && !out_scale)) return CSA_ERR_NULL;
  if (out_dtype != cfg->act && out_dtype != CSA_E4M3) return CSA_ERR_DTYPE;
  if (!aligned16(o) || !aligned16(pos) || !aligned16(out) || (out_scale && !aligned16(out_scale))) return CSA_ERR_ALIGN;
  if (rows < 0 || cfg->d < 8 || cfg->d > 1024 || (cfg->d & 7) || rope_dims < 0 || rope_dims > cfg->d ||
      rope_dims > kMaxRopeDims || (rope_dims & 1) ||
      (rope_dims > 0 && !(rope_theta > 1.f && std::isfinite(rope_theta))) || rows * cfg->H >= (int64_t(1) << 40))
    return CSA_ERR_SHAPE;
  InvRopeArgs a{};
  a.o = o;
  a.rows = rows;
  a.heads = cfg->H;
  a.dim = cfg->d;
  a.pos = pos;
  a.rope_dims = rope_dims;
  a.theta = rope_theta;
  if (rope_dims > 0) make_rope_table(rope_theta, rope_dims, &a.tab);
  a.bf16 = cfg->act == CSA_BF16;
  a.out = out;
  a.e4m3 = out_dtype == CSA_E4M3;
  a.out_scale = out_scale;
  return launch_status(launch_inv_rope_quant(a, reinterpret_cast<cudaStream_t>(stream)));
}

static csa_status indexer_scores_impl(const csa_config* cfg, const void* qI, const float* w, int32_t T, const int64_t* q_pos,
                               const void* kI, const void* kscale, int64_t E_cap, const int32_t* cand, int32_t n_cand,
                               void* scores, int64_t ld_scores, void* ws, size_t ws_bytes, csa_stream_t stream,
                               bool bf16) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!qI || !w || !q_pos || !kI || !scores) return CSA_ERR_NULL;
  if ((st = check_keys(cfg, kI, kscale, E_cap)) != CSA_OK) return st;
  if (!aligned16(qI) || !aligned16(w) || !aligned16(q_pos) || !aligned16(kI) || !aligned16(scores) ||
      (kscale && !aligned16(kscale)) || (cand && !aligned16(cand)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  const int64_t n_cols = cand ? n_cand : E_cap;
  if (T < 0 || E_cap < 0 || (cand && n_cand < 0) || ld_scores < n_cols || cfg->HI > 128 ||
      E_cap * cfg->B >= (int64_t(1) << 31))
    return CSA_ERR_SHAPE;
  IndexerArgs a{};
  a.ws = ws;
  a.qI = qI;
  a.w = w;
  a.q_pos = q_pos;
  a.kI = kI;
  a.kscale = kscale;
  a.cand = cand;
  a.n_cand = n_cand;
  a.scores = static_cast<float*>(scores);
  a.scores_bf16 = bf16;
  a.ld = ld_scores;
  a.B = cfg->B;
  a.T = T;
  a.HI = cfg->HI;
  a.dI = cfg->dI;
  a.m = cfg->m;
  a.E_cap = E_cap;
  a.act = cfg->act;
  a.kidx = cfg->kidx;
  a.num_sms = device_sm_count();
  const size_t need = indexer_workspace_bytes(a);
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  a.err = err_word_ptr();
  return launch_status(launch_indexer(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_indexer_scores(const csa_config* cfg, const void* qI, const float* w, int32_t T,
                              const int64_t* q_pos, const void* kI, const void* kscale, int64_t E_cap,
                              const int32_t* cand, int32_t n_cand, float* scores, int64_t ld_scores, void* ws,
                              size_t ws_bytes, csa_stream_t stream) {
  return indexer_scores_impl(cfg, qI, w, T, q_pos, kI, kscale, E_cap, cand, n_cand, scores, ld_scores, ws, ws_bytes,
                             stream, false);
}

csa_status csa_indexer_scores_bf16(const csa_config* cfg, const void* qI, const float* w, int32_t T,
                                   const int64_t* q_pos, const void* kI, const void* kscale, int64_t E_cap,
                                   const int32_t* cand, int32_t n_cand, void* scores, int64_t ld_scores, void* ws,
                                   size_t ws_bytes, csa_stream_t stream) {
  return indexer_scores_impl(cfg, qI, w, T, q_pos, kI, kscale, E_cap, cand, n_cand, scores, ld_scores, ws, ws_bytes,
                             stream, true);
}

static csa_status indexer_topk_impl(const csa_config* cfg, const void* qI, const float* w, int32_t T, const int64_t* q_pos,
                             const void* kI, const void* kscale, int64_t E_cap, int32_t* idx, void* ws,
                             size_t ws_bytes, csa_stream_t stream, bool bf16) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!qI || !w || !q_pos || !kI || !idx) return CSA_ERR_NULL;
  if ((st = check_keys(cfg, kI, kscale, E_cap)) != CSA_OK) return st;
  if (!aligned16(qI) || !aligned16(w) || !aligned16(q_pos) || !aligned16(kI) || !aligned16(idx) ||
      (kscale && !aligned16(kscale)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (T < 0 || E_cap < 1 || E_cap > (int64_t(1) << 24) || cfg->HI > 128 || E_cap * cfg->B >= (int64_t(1) << 31) ||
      static_cast<int64_t>(cfg->B) * T * E_cap >= (int64_t(1) << 40))
    return CSA_ERR_SHAPE;
  const int64_t rows = static_cast<int64_t>(cfg->B) * T;
  if (rows == 0) return CSA_OK;
  const int sms = device_sm_count();
  const size_t need = indexer_topk_ws(cfg, T, E_cap, sms, bf16);
  if (!ws || ws_bytes < need) return CSA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  IndexerArgs a = indexer_shape(cfg, T, E_cap, sms);
  a.qI = qI;
  a.w = w;
  a.q_pos = q_pos;
  a.kI = kI;
  a.kscale = kscale;
  a.err = err_word_ptr();
  uint8_t* p = static_cast<uint8_t*>(ws);
  a.ws = p;
  p += align_up(indexer_workspace_bytes(a), 256);
  const size_t per_row = align_up(static_cast<size_t>(rows) * 4, 256);
  float* scores = reinterpret_cast<float*>(p);  // fp32, or BF16 (2 bytes a score)
  p += align_up(static_cast<size_t>(rows * E_cap) * (bf16 ? 2 : 4), 256);
  int32_t* nv = reinterpret_cast<int32_t*>(p);
  p += per_row;
  a.scores = scores;
  a.scores_bf16 = bf16;
  a.ld = E_cap;
  a.nv_out = nv;
  cudaError_t e = launch_indexer(a, s);
  if (e != cudaSuccess) return launch_status(e);
  TopkArgs t{};
  t.scores = scores;
  t.ld = E_cap;
  t.rows = rows;
  t.n_cols = E_cap;
  t.n_valid = nv;
  t.cand = nullptr;
  t.k = cfg->k;
  t.idx = idx;
  t.ws = p;
  t.ws_bytes = ws_bytes - static_cast<size_t>(p - static_cast<uint8_t*>(ws));
  t.err = a.err;
  t.num_sms = sms;
  t.bf16 = bf16;
  return launch_status(launch_topk(t, s));
}

csa_status csa_indexer_topk(const csa_config* cfg, const void* qI, const float* w, int32_t T, const int64_t* q_pos,
                            const void* kI, const void* kscale, int64_t E_cap, int32_t* idx, void* ws,
                            size_t ws_bytes, csa_stream_t stream) {
  return indexer_topk_impl(cfg, qI, w, T, q_pos, kI, kscale, E_cap, idx, ws, ws_bytes, stream, false);
}

csa_status csa_indexer_topk_bf16(const csa_config* cfg, const void* qI, const float* w, int32_t T,
                                 const int64_t* q_pos, const void* kI, const void* kscale, int64_t E_cap, int32_t* idx,
                                 void* ws, size_t ws_bytes, csa_stream_t stream) {
  return indexer_topk_impl(cfg, qI, w, T, q_pos, kI, kscale, E_cap, idx, ws, ws_bytes, stream, true);
}

static csa_status topk_impl(const csa_config* cfg, const void* scores, int64_t ld, int64_t rows, int64_t n_cols,
                     const int32_t* n_valid, const int32_t* cand, int32_t* idx, void* ws, size_t ws_bytes,
                     csa_stream_t stream, bool bf16) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!scores || !idx) return CSA_ERR_NULL;
  if (!aligned16(scores) || !aligned16(idx) || (n_valid && !aligned16(n_valid)) || (cand && !aligned16(cand)) ||
      (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (rows < 0 || n_cols < 0 || ld < n_cols || n_cols > (int64_t(1) << 24) || rows > 65535) return CSA_ERR_SHAPE;
  const int sms = device_sm_count();
  const size_t need = topk_workspace_bytes(rows, n_cols, cfg->k, sms, bf16);
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  TopkArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.rows = rows;
  a.n_cols = n_cols;
  a.n_valid = n_valid;
  a.cand = cand;
  a.k = cfg->k;
  a.idx = idx;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.err = err_word_ptr();
  a.num_sms = sms;
  a.bf16 = bf16;
  return launch_status(launch_topk(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_topk(const csa_config* cfg, const float* scores, int64_t ld, int64_t rows, int64_t n_cols,
                    const int32_t* n_valid, const int32_t* cand, int32_t* idx, void* ws, size_t ws_bytes,
                    csa_stream_t stream) {
  return topk_impl(cfg, scores, ld, rows, n_cols, n_valid, cand, idx, ws, ws_bytes, stream, false);
}

csa_status csa_topk_bf16(const csa_config* cfg, const void* scores, int64_t ld, int64_t rows, int64_t n_cols,
                         const int32_t* n_valid, const int32_t* cand, int32_t* idx, void* ws, size_t ws_bytes,
                         csa_stream_t stream) {
  return topk_impl(cfg, scores, ld, rows, n_cols, n_valid, cand, idx, ws, ws_bytes, stream, true);
}

csa_status csa_block_pool(const csa_config* cfg, const float* scores, int64_t ld, int64_t rows, int64_t n_cols,
                          const int32_t* n_valid, int32_t block, int32_t n_blocks, int32_t* pool,
                          int32_t* pool_count, void* ws, size_t ws_bytes, csa_stream_t stream) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!scores || !pool) return CSA_ERR_NULL;
  if (!aligned16(scores) || !aligned16(pool) || (n_valid && !aligned16(n_valid)) ||
      (pool_count && !aligned16(pool_count)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (rows < 0 || n_cols < 0 || ld < n_cols || block < 1 || n_blocks < 1 || n_blocks > 4096 ||
      n_cols > (int64_t(1) << 24) || rows > 65535 || static_cast<int64_t>(block) * n_blocks > (int64_t(1) << 24))
    return CSA_ERR_SHAPE;
  const int sms = device_sm_count();
  const size_t need = pool_workspace_bytes(rows, n_cols, block, n_blocks, sms);
  if (!ws || ws_bytes < need) return CSA_ERR_WORKSPACE;
  PoolArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.rows = rows;
  a.n_cols = n_cols;
  a.n_valid = n_valid;
  a.block = block;
  a.n_blocks = n_blocks;
  a.pool = pool;
  a.pool_count = pool_count;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.err = err_word_ptr();
  a.num_sms = sms;
  return launch_status(launch_block_pool(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_sparse_attn(const csa_config* cfg, const void* q, int32_t T, const void* kv_comp, int64_t E_cap,
                           const int32_t* idx, const void* kv_local, int64_t L, const int64_t* local_base,
                           const int64_t* q_pos, const float* sink, void* out, float* lse, void* ws,
                           size_t ws_bytes, csa_stream_t stream) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!q || !kv_comp || !idx || !kv_local || !local_base || !q_pos || !sink || !out) return CSA_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv_comp) || !aligned16(idx) || !aligned16(kv_local) || !aligned16(local_base) ||
      !aligned16(q_pos) || !aligned16(sink) || !aligned16(out) || (lse && !aligned16(lse)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (T < 0 || E_cap < 0 || L < 0 || !attn_shape_ok(cfg)) return CSA_ERR_SHAPE;
  const int sms = device_sm_count();
  const size_t need = attn_workspace_bytes(cfg->B, T, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms);
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  AttnArgs a{};
  a.q = q;
  a.kv_comp = kv_comp;
  a.idx = idx;
  a.kv_local = kv_local;
  a.local_base = local_base;
  a.q_pos = q_pos;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.B = cfg->B;
  a.T = T;
  a.H = cfg->H;
  a.d = cfg->d;
  a.k = cfg->k;
  a.W = cfg->W;
  a.E_cap = E_cap;
  a.L = L;
  a.softmax_scale = cfg->softmax_scale;
  a.act = cfg->act;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.err = err_word_ptr();
  a.num_sms = sms;
  return launch_status(launch_attn(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_sparse_attn_fp8kv(const csa_config* cfg, const void* q, int32_t T, const void* kv_comp, int64_t E_cap,
                           const int32_t* idx, const void* kv_local, int64_t L, const int64_t* local_base,
                           const int64_t* q_pos, const float* sink, void* out, float* lse, void* ws,
                           size_t ws_bytes, csa_stream_t stream) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!q || !kv_comp || !idx || !kv_local || !local_base || !q_pos || !sink || !out) return CSA_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv_comp) || !aligned16(idx) || !aligned16(kv_local) || !aligned16(local_base) ||
      !aligned16(q_pos) || !aligned16(sink) || !aligned16(out) || (lse && !aligned16(lse)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  const int sms = device_sm_count();
  if (T < 0 || E_cap < 0 || L < 0 || !attn_shape_ok(cfg) || E_cap * cfg->B >= (int64_t(1) << 31) ||
      !attn_quantkv_supported(cfg->B, T, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms))
    return CSA_ERR_SHAPE;
  const size_t need = attn_workspace_bytes(cfg->B, T, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms);
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  AttnArgs a{};
  a.q = q;
  a.kv_comp = kv_comp;
  a.idx = idx;
  a.kv_local = kv_local;
  a.local_base = local_base;
  a.q_pos = q_pos;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.B = cfg->B;
  a.T = T;
  a.H = cfg->H;
  a.d = cfg->d;
  a.k = cfg->k;
  a.W = cfg->W;
  a.E_cap = E_cap;
  a.L = L;
  a.softmax_scale = cfg->softmax_scale;
  a.act = cfg->act;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.err = err_word_ptr();
  a.num_sms = sms;
  return launch_status(launch_attn_fp8kv(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_sparse_attn_mxfp4kv(const csa_config* cfg, const void* q, int32_t T, const void* kv_comp, int64_t E_cap,
                           const int32_t* idx, const void* kv_local, int64_t L, const int64_t* local_base,
                           const int64_t* q_pos, const float* sink, void* out, float* lse, void* ws,
                           size_t ws_bytes, csa_stream_t stream) {
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!q || !kv_comp || !idx || !kv_local || !local_base || !q_pos || !sink || !out) return CSA_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv_comp) || !aligned16(idx) || !aligned16(kv_local) || !aligned16(local_base) ||
      !aligned16(q_pos) || !aligned16(sink) || !aligned16(out) || (lse && !aligned16(lse)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  const int sms = device_sm_count();
  if (T < 0 || E_cap < 0 || L < 0 || !attn_shape_ok(cfg) || E_cap * cfg->B >= (int64_t(1) << 31) ||
      !attn_quantkv_supported(cfg->B, T, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms))
    return CSA_ERR_SHAPE;
  const size_t need = attn_workspace_bytes(cfg->B, T, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms);
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  AttnArgs a{};
  a.q = q;
  a.kv_comp = kv_comp;
  a.idx = idx;
  a.kv_local = kv_local;
  a.local_base = local_base;
  a.q_pos = q_pos;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.B = cfg->B;
  a.T = T;
  a.H = cfg->H;
  a.d = cfg->d;
  a.k = cfg->k;
  a.W = cfg->W;
  a.E_cap = E_cap;
  a.L = L;
  a.softmax_scale = cfg->softmax_scale;
  a.act = cfg->act;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.err = err_word_ptr();
  a.num_sms = sms;
  return launch_status(launch_attn_mxfp4kv(a, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
AttnArgs dense_args(const csa_config* cfg, const void* q, int32_t T, const void* kv_comp, int64_t E_cap,
                    const void* kv_local, int64_t L, const int64_t* local_base, const int64_t* q_pos,
                    const float* sink, void* out, float* lse, void* ws, size_t ws_bytes) {
  AttnArgs a{};
  a.q = q;
  a.kv_comp = kv_comp;
  a.idx = nullptr;
  a.kv_local = kv_local;
  a.local_base = local_base;
  a.q_pos = q_pos;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.B = cfg->B;
  a.T = T;
  a.H = cfg->H;
  a.d = cfg->d;
  a.k = 1;
  a.W = cfg->W;
  a.E_cap = E_cap;
  a.L = L;
  a.softmax_scale = cfg->softmax_scale;
  a.act = cfg->act;
  a.dense_m = cfg->m;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.err = err_word_ptr();
  a.num_sms = device_sm_count();
  return a;
}
}  // namespace

csa_status csa_dense_attn(const csa_config* cfg, const void* q, int32_t T, const void* kv_comp, int64_t E_cap,
                          const void* kv_local, int64_t L, const int64_t* local_base, const int64_t* q_pos,
                          const float* sink, void* out, float* lse, void* ws, size_t ws_bytes, csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!q || !kv_comp || !kv_local || !local_base || !q_pos || !sink || !out) return CSA_ERR_NULL;
  if (!aligned16(q) || !aligned16(kv_comp) || !aligned16(kv_local) || !aligned16(local_base) || !aligned16(q_pos) ||
      !aligned16(sink) || !aligned16(out) || (lse && !aligned16(lse)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (T < 0 || E_cap < 0 || E_cap > (int64_t(1) << 24) || L < 0 || !dense_shape_ok(cfg) ||
      E_cap * cfg->B >= (int64_t(1) << 31))
    return CSA_ERR_SHAPE;
  const size_t need = attn_dense_workspace_bytes(cfg->B, T, cfg->H, cfg->d, E_cap, cfg->W, cfg->act,
                                                 device_sm_count());
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  const AttnArgs a = dense_args(cfg, q, T, kv_comp, E_cap, kv_local, L, local_base, q_pos, sink, out, lse, ws,
                                ws_bytes);
  return launch_status(launch_attn(a, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_hca_decode_step(const csa_config* cfg, const csa_hca_decode_args* d, void* ws, size_t ws_bytes,
                               csa_stream_t stream) {
  csa_status st = check_cfg_hca(cfg);
  if (st != CSA_OK) return st;
  if (!d) return CSA_ERR_NULL;
  if (!d->q_pos || !d->q || !d->sink || !d->kv_comp || !d->kv_tail || !d->z_tail || !d->kv_local ||
      !d->local_base || !d->out)
    return CSA_ERR_NULL;
  const void* ptrs[] = {d->q_pos, d->q, d->sink, d->kv_comp, d->kv_tail, d->z_tail, d->kv_local, d->local_base, d->out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA_ERR_ALIGN;
  if ((d->bias && !aligned16(d->bias)) || (d->lse && !aligned16(d->lse)) || (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (d->E_cap < 1 || d->E_cap > (int64_t(1) << 24) || d->L < 0 || !dense_shape_ok(cfg) || (cfg->d & 1) ||
      d->E_cap * cfg->B >= (int64_t(1) << 31))
    return CSA_ERR_SHAPE;
  const size_t need = attn_dense_workspace_bytes(cfg->B, 1, cfg->H, cfg->d, d->E_cap, cfg->W, cfg->act,
                                                 device_sm_count());
  if (need > 0 && (!ws || ws_bytes < need)) return CSA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Compress1Args c{};
  c.kv = d->kv_tail;
  c.z = d->z_tail;
  c.bias = d->bias;
  c.out = d->kv_comp;
  c.B = cfg->B;
  c.m = cfg->m;
  c.dim = cfg->d;
  c.act_bf16 = cfg->act == CSA_BF16;
  c.q_pos = d->q_pos;
  c.E_cap = d->E_cap;
  cudaError_t e = launch_compress1(c, s);
  if (e != cudaSuccess) return launch_status(e);
  AttnArgs a = dense_args(cfg, d->q, 1, d->kv_comp, d->E_cap, d->kv_local, d->L, d->local_base, d->q_pos,
                          d->sink, d->out, d->lse, ws, ws_bytes);
  a.dense_step = 1;
  return launch_status(launch_attn(a, s));
}

namespace {
csa_status decode_step_impl(const csa_config* cfg, const csa_decode_args* d, void* ws, size_t ws_bytes,
                            csa_stream_t stream, int kv_fmt) {
  const bool qkv = kv_fmt != 0;  // quantised main-KV entries (FP8 or MXFP4): the fused path only
  csa_status st = check_cfg(cfg);
  if (st != CSA_OK) return st;
  if (!d) return CSA_ERR_NULL;
  if (!d->q_pos || !d->q || !d->qI || !d->w || !d->sink || !d->kv_comp || !d->kI || !d->kv_tail || !d->z_tail ||
      !d->kvI_tail || !d->zI_tail || !d->bias || !d->biasI || !d->kv_local || !d->local_base || !d->out)
    return CSA_ERR_NULL;
  if ((st = check_keys(cfg, d->kI, d->kscale, d->E_cap)) != CSA_OK) return st;
  const void* ptrs[] = {d->q_pos, d->q, d->qI, d->w, d->sink, d->kv_comp, d->kI, d->kv_tail, d->z_tail,
                        d->kvI_tail, d->zI_tail, d->bias, d->biasI, d->kv_local, d->local_base, d->out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CSA_ERR_ALIGN;
  if ((d->kscale && !aligned16(d->kscale)) || (d->lse && !aligned16(d->lse)) ||
      (d->idx_out && !aligned16(d->idx_out)) || (d->scores_out && !aligned16(d->scores_out)) ||
      (ws && !aligned16(ws)))
    return CSA_ERR_ALIGN;
  if (d->E_cap < 1 || d->E_cap > (int64_t(1) << 24) || d->L < 0 || !attn_shape_ok(cfg) || cfg->d > 512 || cfg->m > 16 ||
      cfg->HI > 128 || d->E_cap * cfg->B >= (int64_t(1) << 31))
    return CSA_ERR_SHAPE;
  const int sms = device_sm_count();
  if (qkv && !(cfg->act == CSA_BF16 && cfg->d == 512 && cfg->m <= 8 &&
                attn_fp8kv_supported(cfg->B, 1, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms)))
    return CSA_ERR_SHAPE;
  if (!ws || ws_bytes < decode_ws(cfg, d->E_cap, sms)) return CSA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = err_word_ptr();

  uint8_t* p = static_cast<uint8_t*>(ws);
  uint32_t* hist_cnt = reinterpret_cast<uint32_t*>(p);  // kept across steps (zero before the first)
  p += align_up(decode_state_words(cfg->B) * 4, 256);
  void* q_images = p;
  p += align_up(indexer_workspace_bytes(indexer_shape(cfg, 1, d->E_cap, sms)), 256);
  float* scores = reinterpret_cast<float*>(p);
  p += align_up(static_cast<size_t>(cfg->B) * d->E_cap * 4, 256);
  int32_t* nv = reinterpret_cast<int32_t*>(p);
  p += align_up(static_cast<size_t>(cfg->B) * 4, 256);
  int32_t* idx = reinterpret_cast<int32_t*>(p);
  p += align_up(static_cast<size_t>(cfg->B) * cfg->k * 4, 256);
  // the top-k scratch: the fused selection's candidate lists, or the top-k kernels' workspace
  const size_t topk_ws =
      std::max(topk_workspace_bytes(cfg->B, d->E_cap, cfg->k, sms), topk_hist_workspace_bytes(cfg->B, d->E_cap));
  void* ws_topk = p;
  p += align_up(topk_ws, 256);
  void* ws_attn = p;
  if (d->idx_out) idx = d->idx_out;
  if (d->scores_out) scores = d->scores_out;

  // indexer over the visible entries (the tensor-core path also histograms the scores)
  IndexerArgs ia{};
  ia.qI = d->qI;
  ia.w = d->w;
  ia.q_pos = d->q_pos;
  ia.kI = d->kI;
  ia.kscale = d->kscale;
  ia.scores = scores;
  ia.scores_bf16 = d->bf16_scores != 0;
  ia.ld = d->E_cap;
  ia.B = cfg->B;
  ia.T = 1;
  ia.HI = cfg->HI;
  ia.dI = cfg->dI;
  ia.m = cfg->m;
  ia.E_cap = d->E_cap;
  ia.act = cfg->act;
  ia.kidx = cfg->kidx;
  ia.err = err;
  ia.num_sms = sms;
  ia.nv_out = nv;
  ia.ws = q_images;
  ia.wait_ns = g_debug_wait_ns.load(std::memory_order_relaxed);
  ia.skip_key_loads = g_debug_skip_loads.load(std::memory_order_relaxed) != 0;
  cudaError_t e;
  // the attention on the decode split plan waits for each query's list through the step
  // counters after the histograms and tickets, not for the whole selection kernel
  uint32_t* sel_done = hist_cnt + static_cast<size_t>(cfg->B) * 4160 + cfg->B;
  uint32_t* sel_seen = sel_done + cfg->B;
  uint32_t* sel_chunk_ctr = sel_seen + cfg->B;
  uint32_t* sel_thr = sel_chunk_ctr + cfg->B;  // [B][2]
  bool handoff = false;
  int cand_cap = 0;
  if (indexer_uses_tensor_cores(ia) && cfg->m <= 8) {
    // 1-2. one launch: compression of the completed block (both caches), the query images,
    //      the scores and their histogram; 3. the top-k from that histogram
    handoff = attn_fp8kv_supported(cfg->B, 1, cfg->H, cfg->d, cfg->k, cfg->W, cfg->act, sms);
    DecodeFuse& f = ia.fuse;
    f.on = true;
    f.kv_tail = d->kv_tail;
    f.z_tail = d->z_tail;
    f.bias = d->bias;
    f.kv_comp = d->kv_comp;
    f.d = cfg->d;
    f.kvI_tail = d->kvI_tail;
    f.zI_tail = d->zI_tail;
    f.biasI = d->biasI;
    f.act_bf16 = cfg->act == CSA_BF16;
    f.kv_fmt = kv_fmt;
    f.hist = hist_cnt;
    ia.images_ready = true;
    e = launch_indexer(ia, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    SelHandoff ho{};
    if (handoff) {
      cand_cap = decode_cand_cap(cfg, d->E_cap, sms);
      ho.done = sel_done;
      if (cand_cap > 0) {
        ho.chunks = sel_chunk_ctr;
        ho.thr = sel_thr;
        ho.cand_cap = cand_cap;
      }
      ho.pf_rows = static_cast<const uint8_t*>(d->kv_comp);
      ho.pf_row_bytes = kv_fmt == 1 ? 576 : kv_fmt == 2 ? 288 : static_cast<int64_t>(cfg->d) * 2;
      ho.pf_seq_rows = d->E_cap;
    }
    e = launch_topk_hist(scores, d->E_cap, cfg->B, d->E_cap, nv, hist_cnt, cfg->k, idx, ws_topk, sms, s, nullptr,
                         ia.scores_bf16, ho);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  } else {
    if (qkv) return CSA_ERR_SHAPE;  // quantised entries: the fused path only
    // 1. compress the block the new token completes (main KV, then indexer keys)
    CompressArgs c{};
    c.B = cfg->B;
    c.m = cfg->m;
    c.act_bf16 = cfg->act == CSA_BF16;
    c.q_pos = d->q_pos;
    c.E_cap = d->E_cap;
    c.err = err;
    c.job[0] = CompressJob{d->kv_tail, d->z_tail, d->bias, cfg->d, d->kv_comp, cfg->act, nullptr};
    c.job[1] = CompressJob{d->kvI_tail, d->zI_tail, d->biasI, cfg->dI, d->kI, cfg->kidx, d->kscale};
    c.n_jobs = 2;
    e = launch_compress(c, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    // 2. indexer; 3. top-k
    e = launch_indexer(ia, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    TopkArgs ta{};
    ta.scores = scores;
    ta.ld = d->E_cap;
    ta.rows = cfg->B;
    ta.n_cols = d->E_cap;
    ta.n_valid = nv;
    ta.k = cfg->k;
    ta.idx = idx;
    ta.ws = ws_topk;
    ta.ws_bytes = topk_ws;
    ta.err = err;
    ta.num_sms = sms;
    ta.bf16 = ia.scores_bf16;
    e = launch_topk(ta, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  }

  // 4. sparse attention over the selection plus the window, with the sink
  AttnArgs aa{};
  aa.q = d->q;
  aa.kv_comp = d->kv_comp;
  aa.idx = idx;
  aa.kv_local = d->kv_local;
  aa.local_base = d->local_base;
  aa.q_pos = d->q_pos;
  aa.sink = d->sink;
  aa.out = d->out;
  aa.lse = d->lse;
  aa.B = cfg->B;
  aa.T = 1;
  aa.H = cfg->H;
  aa.d = cfg->d;
  aa.k = cfg->k;
  aa.W = cfg->W;
  aa.E_cap = d->E_cap;
  aa.L = d->L;
  aa.softmax_scale = cfg->softmax_scale;
  aa.act = cfg->act;
  aa.ws = ws_attn;
  aa.err = err;
  aa.num_sms = sms;
  if (handoff) {
    aa.sel_done = sel_done;
    aa.sel_seen = sel_seen;
    if (cand_cap > 0) {
      aa.cand_cap = cand_cap;
      aa.sel_chunks = sel_chunk_ctr;
      aa.sel_thr = sel_thr;
      aa.sel_slots = static_cast<const uint32_t*>(ws_topk);
      aa.sel_n_chunks = sel_chunks(d->E_cap);
      aa.sel_slot_words = sel_slot_words();
      aa.sel_slot_cap = sel_slot_cap();
      aa.min_split = 1 + cand_cap / 128;
    }
  }
  return launch_status(kv_fmt == 2 ? launch_attn_mxfp4kv(aa, s) : kv_fmt == 1 ? launch_attn_fp8kv(aa, s) : launch_attn(aa, s));
}
}  // namespace

csa_status csa_decode_step_reset(const csa_config* cfg, void* ws, size_t ws_bytes, csa_stream_t stream) {
  if (!cfg || !ws) return CSA_ERR_NULL;
  if (cfg->B < 1) return CSA_ERR_SHAPE;
  if (!aligned16(ws)) return CSA_ERR_ALIGN;
  const size_t bytes = decode_state_words(cfg->B) * 4;
  if (ws_bytes < bytes) return CSA_ERR_WORKSPACE;
  return launch_status(cudaMemsetAsync(ws, 0, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

csa_status csa_decode_step(const csa_config* cfg, const csa_decode_args* d, void* ws, size_t ws_bytes,
                           csa_stream_t stream) {
  return decode_step_impl(cfg, d, ws, ws_bytes, stream, 0);
}

csa_status csa_decode_step_fp8kv(const csa_config* cfg, const csa_decode_args* d, void* ws, size_t ws_bytes,
                                 csa_stream_t stream) {
  return decode_step_impl(cfg, d, ws, ws_bytes, stream, 1);
}

csa_status csa_decode_step_mxfp4kv(const csa_config* cfg, const csa_decode_args* d, void* ws, size_t ws_bytes,
                                   csa_stream_t stream) {
  return decode_step_impl(cfg, d, ws, ws_bytes, stream, 2);
}

}  // extern "C"
