// Causal top-k selection and the CSA2 block pool.
//
// "DeepSeek V4-Flash: The Cost of Deciding What to Read", section "The Lightning Indexer":
// a cheap scoring pass keeps the top 512 compressed entries and the attention runs over
// those only.  Order: score descending, position ascending (the lowest position wins a
// tie; -0 equals +0).  Output: the kept positions in ascending order, -1 padded.
//
// Design: a row is cut into chunks; one CTA finds the k best of its chunk by a three-pass
// radix select (11/11/10 bits) over order-preserving uint32 keys held in shared memory,
// then compacts the winners in position order with warp ballots.  The winners of all
// chunks, concatenated in chunk order, are again in ascending position order, so the
// same kernel merges them level by level until one chunk remains.  Every decision is
// exact and independent of scheduling: the result is deterministic.
//
// CSA2 pool ("DeepSeek-V4.1-Flash's KV-Cache Compression ...", section 3, Hierarchical
// Sparse Indexer): block maxima of 8 positions, the same top-k over the block maxima, then
// expansion of the kept blocks to positions.
#include <algorithm>

#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {
namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kHistBins = 2048;
constexpr int kCandChunk = 16384;
constexpr int kRawChunkMax = 8192;
constexpr int kMaxLevels = 8;

struct LevelParams {
  // raw-score input (level 0)
  const float* scores;
  int64_t ld;
  const int32_t* n_valid;
  const int32_t* cand;  // [rows, n_in] position map or null
  // candidate input (levels >= 1): [rows, in_ld] keys and positions (-1 = empty)
  const uint32_t* in_key;
  const int32_t* in_pos;
  int64_t in_ld;
  int64_t n_in;
  int chunk;
  int k;
  uint32_t* out_key;
  int32_t* out_pos;
  int64_t out_ld;
  int32_t* idx;  // final level output [rows, k]
  int final_level;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Radix select of the k-th largest key among keys[0:n) (key 0 = empty slot).  Returns the
// threshold key T and the number `quota` of keys equal to T that belong to the selection.
__device__ void block_select(const uint32_t* keys, int n, int k, uint32_t* hist, uint32_t* tmp,
                             uint32_t* s_res, uint32_t& T, int& quota) {
  const int tid = threadIdx.x, lane = tid & 31;
  // count non-empty keys
  uint32_t cnt = 0;
  for (int e = tid; e < n; e += NT) cnt += keys[e] != 0u;
  uint32_t total;
  block_exclusive_scan<NT>(cnt, tmp, &total);
  if (static_cast<int>(total) <= k) {
    T = 1u;
    quota = 0x7fffffff;
    return;
  }
  uint32_t prefix = 0u, mask = 0u;
  int kk = k;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass], nb = 1 << widths[pass];
    for (int i = tid; i < nb; i += NT) hist[i] = 0u;
    __syncthreads();
    for (int base = 0; base < n; base += NT) {
      const int e = base + tid;
      const uint32_t key = e < n ? keys[e] : 0u;
      const bool part = key != 0u && (key & mask) == prefix;
      const uint32_t digit = part ? ((key >> shift) & static_cast<uint32_t>(nb - 1)) : 0xffffffffu;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (part && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    const int bpt = nb / NT;  // bins per thread (4 or 2)
    const int b0 = tid * bpt;
    uint32_t local = 0;
    for (int q = 0; q < bpt; ++q) local += hist[b0 + q];
    uint32_t tot;
    const uint32_t excl = block_exclusive_scan<NT>(local, tmp, &tot);
    uint32_t run = tot - excl - local;  // keys in bins above this thread's bins
    for (int q = bpt - 1; q >= 0; --q) {
      const uint32_t h = hist[b0 + q];
      if (run < static_cast<uint32_t>(kk) && run + h >= static_cast<uint32_t>(kk)) {
        s_res[0] = static_cast<uint32_t>(b0 + q);
        s_res[1] = run;
      }
      run += h;
    }
    __syncthreads();
    const uint32_t bin = s_res[0];
    kk -= static_cast<int>(s_res[1]);
    prefix |= bin << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    __syncthreads();
  }
  T = prefix;
  quota = kk;
}

template <bool RAW>
__global__ void __launch_bounds__(NT) topk_level_kernel(LevelParams p) {
  extern __shared__ uint32_t sm[];
  const int chunk = p.chunk;
  uint32_t* keys = sm;
  int32_t* spos = reinterpret_cast<int32_t*>(sm + chunk);  // candidate levels only
  uint32_t* hist = sm + chunk * (RAW ? 1 : 2);
  uint32_t* tmp = hist + kHistBins;
  uint32_t* wtot = tmp + 32;  // [3][NW]
  uint32_t* s_res = wtot + 3 * NW;

  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int n = static_cast<int>(std::min<int64_t>(chunk, p.n_in - c0));

  // load the chunk
  if (RAW) {
    int64_t nvr = p.n_valid ? p.n_valid[row] : p.n_in;
    nvr = nvr < p.n_in ? nvr : p.n_in;
    const float* src = p.scores + row * p.ld + c0;
    const int32_t* cmap = p.cand ? p.cand + row * p.n_in + c0 : nullptr;
    for (int e = tid; e < n; e += NT) {
      bool valid = c0 + e < nvr;
      if (valid && cmap) valid = cmap[e] >= 0;
      uint32_t key = 0u;
      if (valid) {
        key = f2key(src[e]);
        if (key == 0u) key = 1u;
      }
      keys[e] = key;
    }
  } else {
    const uint32_t* ks = p.in_key + row * p.in_ld + c0;
    const int32_t* ps = p.in_pos + row * p.in_ld + c0;
    for (int e = tid; e < n; e += NT) {
      const int32_t pos = ps[e];
      keys[e] = pos >= 0 ? ks[e] : 0u;
      spos[e] = pos;
    }
  }
  __syncthreads();

  uint32_t T;
  int quota;
  block_select(keys, n, p.k, hist, tmp, s_res, T, quota);

  // compaction in position order: warp w owns elements [w*seg, (w+1)*seg)
  const int seg = ((n + NW - 1) / NW + 31) & ~31;
  const int lo = warp * seg, hi = std::min(n, lo + seg);
  uint32_t gt = 0, eq = 0;
  for (int base = lo; base < hi; base += 32) {
    const int e = base + lane;
    const uint32_t key = e < hi ? keys[e] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, key != 0u && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, key != 0u && key == T));
  }
  if (lane == 0) {
    wtot[warp] = gt;
    wtot[NW + warp] = eq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t eq_run = 0, sel_run = 0;
    for (int w = 0; w < NW; ++w) {
      const uint32_t g = wtot[w], q = wtot[NW + w];
      const int64_t left = static_cast<int64_t>(quota) - eq_run;
      const uint32_t take = left <= 0 ? 0u : (left >= q ? q : static_cast<uint32_t>(left));
      wtot[NW + w] = eq_run;          // equal keys before warp w
      wtot[2 * NW + w] = sel_run;     // selected before warp w
      eq_run += q;
      sel_run += g + take;
    }
    s_res[2] = sel_run;
  }
  __syncthreads();
  uint32_t eq_before = wtot[NW + warp], out = wtot[2 * NW + warp];
  const uint32_t n_sel = s_res[2];
  for (int base = lo; base < hi; base += 32) {
    const int e = base + lane;
    const uint32_t key = e < hi ? keys[e] : 0u;
    const bool is_eq = key != 0u && key == T;
    const uint32_t eq_bits = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t my_eq_rank = eq_before + __popc(eq_bits & lanemask_lt());
    const bool sel = (key != 0u && key > T) || (is_eq && my_eq_rank < static_cast<uint32_t>(quota));
    const uint32_t sel_bits = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const uint32_t o = out + __popc(sel_bits & lanemask_lt());
      int32_t pos;
      if (RAW) {
        pos = p.cand ? p.cand[row * p.n_in + c0 + e] : static_cast<int32_t>(c0 + e);
      } else {
        pos = spos[e];
      }
      if (p.final_level) {
        p.idx[row * p.k + o] = pos;
      } else {
        const int64_t slot = row * p.out_ld + static_cast<int64_t>(blockIdx.x) * p.k + o;
        p.out_key[slot] = key;
        p.out_pos[slot] = pos;
      }
    }
    out += __popc(sel_bits);
    eq_before += __popc(eq_bits);
  }
  // pad the k slots
  for (int o = static_cast<int>(n_sel) + tid; o < p.k; o += NT) {
    if (p.final_level) {
      p.idx[row * p.k + o] = -1;
    } else {
      const int64_t slot = row * p.out_ld + static_cast<int64_t>(blockIdx.x) * p.k + o;
      p.out_key[slot] = 0u;
      p.out_pos[slot] = -1;
    }
  }
}

struct Plan {
  int nlev;
  int64_t n_in[kMaxLevels];
  int chunk[kMaxLevels];
  int64_t n_chunks[kMaxLevels];
};

Plan make_plan(int64_t rows, int64_t n_cols, int k, int num_sms) {
  Plan pl{};
  int c0 = 8192;
  while (c0 > 2048 && c0 / 2 >= 2 * k && rows * ((n_cols + c0 - 1) / c0) < 2 * num_sms) c0 /= 2;
  if (c0 < 2 * k) c0 = std::max(c0, 2 * k);
  int64_t n_in = n_cols;
  int lev = 0;
  int chunk = c0;
  while (true) {
    pl.n_in[lev] = n_in;
    pl.chunk[lev] = chunk;
    pl.n_chunks[lev] = (n_in + chunk - 1) / chunk;
    if (pl.n_chunks[lev] <= 1 || lev + 1 >= kMaxLevels) {
      pl.n_chunks[lev] = 1;
      pl.chunk[lev] = static_cast<int>(n_in);
      ++lev;
      break;
    }
    n_in = pl.n_chunks[lev] * k;
    chunk = kCandChunk;
    ++lev;
  }
  pl.nlev = lev;
  return pl;
}

size_t level_smem(int chunk, bool raw) {
  return (static_cast<size_t>(chunk) * (raw ? 1 : 2) + kHistBins + 32 + 3 * NW + 4) * 4;
}

// Block maxima of a row (4 consecutive blocks per thread); with `hist`, also the row's
// histogram of their order-preserving keys (4096 bins of key >> 20, added to a zeroed row of
// kTopkHistRowWords words) for the histogram-guided top-k.
constexpr int kBmaxPer = 4;
constexpr int kBmaxThreads = 256;

__global__ void __launch_bounds__(kBmaxThreads) blockmax_kernel(const float* scores, int64_t ld, int64_t n_cols,
                                                                const int32_t* n_valid, int block, float* bmax,
                                                                int64_t ld_b, int32_t* nb_out, uint32_t* hist) {
  __shared__ uint32_t h[kTopkHistBins];
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.y;
  int64_t nv = n_valid ? n_valid[row] : n_cols;
  nv = nv < n_cols ? nv : n_cols;
  nv = nv < 0 ? 0 : nv;
  const int64_t nb = (nv + block - 1) / block;
  if (blockIdx.x == 0 && threadIdx.x == 0) nb_out[row] = static_cast<int32_t>(nb);
  if (hist) {
    for (int i = threadIdx.x; i < kTopkHistBins; i += kBmaxThreads) h[i] = 0u;
    __syncthreads();
  }
  const float* srow = scores + row * ld;
  const int64_t j0 = (static_cast<int64_t>(blockIdx.x) * kBmaxThreads + threadIdx.x) * kBmaxPer;
  float m[kBmaxPer];
  const bool vec = block == 8 && j0 + kBmaxPer <= nb && (j0 + kBmaxPer) * 8 <= nv &&
                   (reinterpret_cast<uintptr_t>(srow + j0 * 8) & 15) == 0;
  if (vec) {
    float4 x[2 * kBmaxPer];
#pragma unroll
    for (int u = 0; u < 2 * kBmaxPer; ++u) x[u] = __ldcg(reinterpret_cast<const float4*>(srow + j0 * 8) + u);
#pragma unroll
    for (int u = 0; u < kBmaxPer; ++u) {
      const float4 a = x[2 * u], b = x[2 * u + 1];
      m[u] = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
    }
  } else {
#pragma unroll
    for (int u = 0; u < kBmaxPer; ++u) {
      const int64_t j = j0 + u;
      m[u] = -INFINITY;
      if (j < nb) {
        const int64_t hi = std::min<int64_t>((j + 1) * block, nv);
        for (int64_t p = j * block; p < hi; ++p) m[u] = fmaxf(m[u], srow[p]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kBmaxPer; ++u) {
    const int64_t j = j0 + u;
    if (j < nb) {
      bmax[row * ld_b + j] = m[u];
      if (hist) atomicAdd(&h[f2key(m[u]) >> 20], 1u);
    }
  }
  if (hist) {
    __syncthreads();
    uint32_t* rh = hist + row * kTopkHistRowWords;
    for (int i = threadIdx.x; i < kTopkHistBins; i += kBmaxThreads)
      if (h[i]) atomicAdd(&rh[i], h[i]);
  }
}

// Expands the kept blocks (ascending, -1 padded) to their visible positions: thread t of the
// row's grid writes slots 4t..4t+3.  The top-k keeps exactly min(n_blocks, nb) blocks, and only
// the row's last block (index nb - 1, then last in ascending order) can be partial, so the
// pool's size follows without a reduction.
__global__ void pool_expand_kernel(const int32_t* sel, int n_blocks, int block, const int32_t* n_valid,
                                   int64_t n_cols, int32_t* pool, int32_t* pool_count) {
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.y;
  int64_t nv = n_valid ? n_valid[row] : n_cols;
  nv = nv < n_cols ? nv : n_cols;
  nv = nv < 0 ? 0 : nv;
  const int64_t width = static_cast<int64_t>(n_blocks) * block;
  const int32_t* srow = sel + row * n_blocks;
  const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i0 < width) {
    int32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u;
      o[u] = -1;
      if (i < width) {
        const int32_t j = __ldg(srow + i / block);
        const int64_t ppos = static_cast<int64_t>(j) * block + i % block;
        if (j >= 0 && ppos < nv) o[u] = static_cast<int32_t>(ppos);
      }
    }
    int32_t* dst = pool + row * width + i0;
    if ((width & 3) == 0) {
      *reinterpret_cast<int4*>(dst) = make_int4(o[0], o[1], o[2], o[3]);
    } else {
      for (int u = 0; u < 4 && i0 + u < width; ++u) dst[u] = o[u];
    }
  }
  if (pool_count && blockIdx.x == 0 && threadIdx.x == 0) {
    const int64_t nb = (nv + block - 1) / block;
    const int64_t n_sel = nb < n_blocks ? nb : n_blocks;
    int64_t cnt = n_sel * block;
    if (n_sel > 0 && srow[n_sel - 1] == nb - 1) cnt -= nb * block - nv;
    pool_count[row] = static_cast<int32_t>(cnt);
  }
}

cudaError_t run_levels(const Plan& pl, const float* scores, int64_t ld, int64_t rows, const int32_t* n_valid,
                       const int32_t* cand, int k, int32_t* idx, uint8_t* ws, cudaStream_t s) {
  // ping-pong candidate buffers sized for the widest intermediate level
  int64_t max_slots = 0;
  for (int l = 0; l + 1 < pl.nlev; ++l) max_slots = std::max<int64_t>(max_slots, pl.n_chunks[l] * k);
  const size_t buf = align_up(static_cast<size_t>(rows * max_slots) * 4, 256);
  uint32_t* key[2] = {reinterpret_cast<uint32_t*>(ws), reinterpret_cast<uint32_t*>(ws + 2 * buf)};
  int32_t* pos[2] = {reinterpret_cast<int32_t*>(ws + buf), reinterpret_cast<int32_t*>(ws + 3 * buf)};
  for (int l = 0; l < pl.nlev; ++l) {
    LevelParams p{};
    p.scores = scores;
    p.ld = ld;
    p.n_valid = n_valid;
    p.cand = cand;
    p.n_in = pl.n_in[l];
    p.chunk = pl.chunk[l];
    p.k = k;
    p.final_level = (l == pl.nlev - 1);
    p.idx = idx;
    if (l > 0) {
      p.in_key = key[(l - 1) & 1];
      p.in_pos = pos[(l - 1) & 1];
      p.in_ld = max_slots;
    }
    if (!p.final_level) {
      p.out_key = key[l & 1];
      p.out_pos = pos[l & 1];
      p.out_ld = max_slots;
    }
    dim3 grid(static_cast<unsigned>(pl.n_chunks[l]), static_cast<unsigned>(rows));
    const size_t smem = level_smem(p.chunk, l == 0);
    static std::atomic<unsigned long long> attr_set{0};  // both instantiations, largest chunk
    if (first_use_in_context(attr_set)) {
      cudaFuncSetAttribute(topk_level_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(level_smem(kRawChunkMax, true)));
      cudaFuncSetAttribute(topk_level_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(level_smem(kCandChunk, false)));
    }
    cudaError_t e = (l == 0) ? launch_pdl(topk_level_kernel<true>, grid, dim3(NT), smem, s, p)
                             : launch_pdl(topk_level_kernel<false>, grid, dim3(NT), smem, s, p);
    count_launches(1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t levels_ws(const Plan& pl, int64_t rows, int k) {
  int64_t max_slots = 0;
  for (int l = 0; l + 1 < pl.nlev; ++l) max_slots = std::max<int64_t>(max_slots, pl.n_chunks[l] * k);
  return 4 * align_up(static_cast<size_t>(rows * max_slots) * 4, 256);
}

}  // namespace

size_t topk_workspace_bytes(int64_t rows, int64_t n_cols, int k, int num_sms, bool bf16) {
  // the scratch of the path launch_topk takes: the histogram path's counts and slots, none for
  // the row kernel (shared memory only; BF16 rows of any length), else the level path's
  // ping-pong candidate buffers
  if (topk_uses_hist(rows, n_cols, false)) return topk_hist_standalone_bytes(rows, n_cols);
  if (bf16 || topk_uses_rows(rows, n_cols, false, k)) return 0;
  return levels_ws(make_plan(rows, n_cols, k, num_sms), rows, k);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  if (topk_uses_hist(a.rows, a.n_cols, a.cand != nullptr)) return launch_topk_hist_standalone(a, s);
  if (a.bf16 || topk_uses_rows(a.rows, a.n_cols, a.cand != nullptr, a.k))
    return launch_topk_rows(a.scores, a.ld, a.rows, a.n_cols, a.n_valid, a.k, a.idx, s, a.cand, a.bf16);
  const Plan pl = make_plan(a.rows, std::max<int64_t>(a.n_cols, 1), a.k, a.num_sms);
  return run_levels(pl, static_cast<const float*>(a.scores), a.ld, a.rows, a.n_valid, a.cand, a.k, a.idx,
                    static_cast<uint8_t*>(a.ws), s);
}

size_t pool_workspace_bytes(int64_t rows, int64_t n_cols, int block, int n_blocks, int num_sms) {
  const int64_t nbmax = (n_cols + block - 1) / block;
  const size_t bm = align_up(static_cast<size_t>(rows * std::max<int64_t>(nbmax, 1)) * 4, 256);
  const size_t nb = align_up(static_cast<size_t>(rows) * 4, 256);
  const size_t sel = align_up(static_cast<size_t>(rows) * n_blocks * 4, 256);
  const size_t rest = topk_uses_hist(rows, std::max<int64_t>(nbmax, 1), false)
                          ? topk_hist_standalone_bytes(rows, std::max<int64_t>(nbmax, 1))
                          : levels_ws(make_plan(rows, std::max<int64_t>(nbmax, 1), n_blocks, num_sms), rows, n_blocks);
  return bm + nb + sel + rest;
}

cudaError_t launch_block_pool(const PoolArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const int64_t nbmax = std::max<int64_t>((a.n_cols + a.block - 1) / a.block, 1);
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  float* bmax = reinterpret_cast<float*>(ws);
  ws += align_up(static_cast<size_t>(a.rows * nbmax) * 4, 256);
  int32_t* nb = reinterpret_cast<int32_t*>(ws);
  ws += align_up(static_cast<size_t>(a.rows) * 4, 256);
  int32_t* sel = reinterpret_cast<int32_t*>(ws);
  ws += align_up(static_cast<size_t>(a.rows) * a.n_blocks * 4, 256);
  // few rows of many blocks: the block maxima are histogrammed as they are made, and the
  // histogram-guided top-k (several CTAs per row) selects the blocks
  const bool by_hist = topk_uses_hist(a.rows, nbmax, false);
  uint32_t* hist = nullptr;
  cudaError_t e = cudaSuccess;
  if (by_hist) {
    hist = reinterpret_cast<uint32_t*>(ws);
    e = cudaMemsetAsync(hist, 0, static_cast<size_t>(a.rows) * (kTopkHistRowWords + 1) * 4, s);
    if (e != cudaSuccess) return e;
  }
  const int64_t per_cta = static_cast<int64_t>(kBmaxThreads) * kBmaxPer;
  dim3 g1(static_cast<unsigned>((nbmax + per_cta - 1) / per_cta), static_cast<unsigned>(a.rows));
  e = launch_pdl(blockmax_kernel, g1, dim3(kBmaxThreads), 0, s, a.scores, a.ld, a.n_cols, a.n_valid, a.block, bmax,
                 static_cast<int64_t>(nbmax), nb, hist);
  count_launches(1);
  if (e != cudaSuccess) return e;
  if (by_hist) {
    const size_t hbytes = align_up(static_cast<size_t>(a.rows) * (kTopkHistRowWords + 1) * 4, 256);
    e = launch_topk_hist(bmax, nbmax, a.rows, nbmax, nb, hist, a.n_blocks, sel, ws + hbytes, a.num_sms, s);
  } else if (topk_uses_rows(a.rows, nbmax, false, a.n_blocks)) {
    e = launch_topk_rows(bmax, nbmax, a.rows, nbmax, nb, a.n_blocks, sel, s);
  } else {
    const Plan pl = make_plan(a.rows, nbmax, a.n_blocks, a.num_sms);
    e = run_levels(pl, bmax, nbmax, a.rows, nb, nullptr, a.n_blocks, sel, ws, s);
  }
  if (e != cudaSuccess) return e;
  const int32_t* csel = sel;
  const int64_t width = static_cast<int64_t>(a.n_blocks) * a.block;
  const dim3 ge(static_cast<unsigned>((width + 1023) / 1024), static_cast<unsigned>(a.rows));
  e = launch_pdl(pool_expand_kernel, ge, dim3(256), 0, s, csel, a.n_blocks, a.block, a.n_valid, a.n_cols, a.pool,
                 a.pool_count);
  count_launches(1);
  return e;
}

}  // namespace csa

