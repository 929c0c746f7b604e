// csa_topk_noalloc: the top-k of csa_topk for callers that cannot allocate device memory.
//
// Some callers only ever receive input and output buffers: for example a plugin running
// inside another runtime that owns every device allocation, or code on a latency-critical
// path where a device allocation could block or fail.  They cannot hand csa_topk a workspace.
// This entry point uses a fixed scratch array that lives in the library itself (a file-scope
// __device__ array of CSA_NOALLOC_SCRATCH_BYTES, resident on every GPU that loads the library
// until the process exits) and allocates nothing.
//
// The array's name in host code is only a host-side stand-in for the device object, so its
// device address is looked up with cudaGetSymbolAddress and passed to the kernels.  The
// lookup runs on the first call in each CUDA context (with that context's device current) and
// again whenever the current context changes (a device reset or a new primary context loads
// the module again, at a new address); the address is cached per device with the id of the
// context it belongs to.  Every call shares the one array and finds it as the previous call
// left it: whatever must start at zero is cleared on the stream before use, and two calls
// whose work overlaps on the GPU race on it.
#include <mutex>

#include "csa_internal.h"

namespace {

constexpr size_t kScratchBytes = CSA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
struct ScratchSlot {
  unsigned long long ctx;  // id of the context the address belongs to
  void* ptr;
};
ScratchSlot g_scratch[kMaxDev] = {};

// Device address of the scratch array in the current context.
csa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return CSA_ERR_CUDA;
  const unsigned long long id = csa::current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch[dev].ptr || id == 0 || g_scratch[dev].ctx != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return CSA_ERR_CUDA;
    g_scratch[dev] = ScratchSlot{csa::current_context_id(), p};
  }
  *out = g_scratch[dev].ptr;
  return CSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" csa_status csa_topk_noalloc(const csa_config* cfg, const float* scores, int64_t ld, int64_t rows,
                                       int64_t n_cols, const int32_t* n_valid, const int32_t* cand, int32_t* idx,
                                       csa_stream_t stream) {
  if (!cfg || !scores || !idx) return CSA_ERR_NULL;
  if (cfg->k < 1 || cfg->k > 4096) return CSA_ERR_SHAPE;
  if (!aligned16(scores) || !aligned16(idx) || (n_valid && !aligned16(n_valid)) || (cand && !aligned16(cand)))
    return CSA_ERR_ALIGN;
  if (rows < 0 || n_cols < 0 || ld < n_cols || n_cols > (int64_t(1) << 24) || rows > 65535) return CSA_ERR_SHAPE;
  const int sms = csa::device_sm_count();
  if (csa::topk_workspace_bytes(rows, n_cols, cfg->k, sms) > kScratchBytes) return CSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const csa_status st = scratch_address(&scratch);
  if (st != CSA_OK) return st;
  csa::TopkArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.rows = rows;
  a.n_cols = n_cols;
  a.n_valid = n_valid;
  a.cand = cand;
  a.k = cfg->k;
  a.idx = idx;
  a.ws = scratch;
  a.ws_bytes = kScratchBytes;
  a.num_sms = sms;
  return csa::launch_topk(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
