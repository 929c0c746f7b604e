// Histogram-guided top-k for a few long rows (the decode step).
//
// Same contract as the chunked top-k ("DeepSeek V4-Flash: The Cost of Deciding What to
// Read", section "The Lightning Indexer": keep the k best entries; ties go to the lowest
// position; output ascending, -1 padded).
//
// Every visible score of row r is counted in a two-level histogram of its order-preserving
// key: 4096 fine bins (key >> 20) and 64 coarse bins (key >> 26).  The decode step fills it
// in the indexer epilogue; the standalone call fills it with topk_hist_build_kernel.  From it,
// the threshold digit b1 is the largest fine bin whose suffix count reaches k, so every one
// of the k best scores has digit >= b1.
//  1. topk_filter_kernel (wide grid) appends every score with digit >= b1 to the row's
//     candidate list (about k plus one bin's worth; order irrelevant).
//  2. topk_final_kernel (one CTA per row) finds the exact k-th key by radix select over the
//     candidates, resolves ties at that key by lowest position, and writes the winners in
//     ascending position with a bucket-counting sort.  If the list overflowed its capacity
//     (a bin full of ties) it selects over the whole row instead, in position order.
#include <algorithm>

#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {
namespace {

constexpr int NT = 512;
constexpr int kFine = kTopkHistBins;     // 4096
constexpr int kCoarse = kTopkHistCoarse; // 64
constexpr int kRowWords = kTopkHistRowWords;
constexpr int kRadixBins = 2048;
constexpr int kSortBuckets = 1024;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int64_t row_valid(const int32_t* n_valid, int64_t row, int64_t n_cols) {
  if (!n_valid) return n_cols;
  const int64_t v = n_valid[row];
  return v < 0 ? 0 : (v < n_cols ? v : n_cols);
}

// One warp: the largest index b of 64 bins (values cnt(b)) whose suffix count reaches `need`;
// returns -1 when the 64 bins hold fewer than `need`, else b and (via *above) the count of
// the bins above b.
__device__ __forceinline__ int warp_suffix_find64(const uint32_t* bins, uint32_t need, uint32_t* above) {
  const int lane = threadIdx.x & 31;
  // lane l owns bins 63-2l and 62-2l (descending), so a prefix scan runs from the top
  const uint32_t c_hi = __ldcg(bins + 63 - 2 * lane);
  const uint32_t c_lo = __ldcg(bins + 62 - 2 * lane);
  const uint32_t mine = c_hi + c_lo;
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t excl = incl - mine;  // count of the bins above this lane's pair
  const uint32_t hit = __ballot_sync(0xffffffffu, incl >= need);
  if (hit == 0u) return -1;
  const int l = __ffs(hit) - 1;  // first lane (from the top) whose inclusive count reaches need
  const uint32_t ex = __shfl_sync(0xffffffffu, excl, l);
  const uint32_t ch = __shfl_sync(0xffffffffu, c_hi, l);
  if (ex + ch >= need) {
    *above = ex;
    return 63 - 2 * l;
  }
  *above = ex + ch;
  return 62 - 2 * l;
}

// Threshold fine digit of a row (warp 0 of the block calls it); 0 when fewer than k scores.
__device__ uint32_t threshold_digit(const uint32_t* row_hist, int k) {
  const uint32_t* fine = row_hist;
  const uint32_t* coarse = row_hist + kFine;
  uint32_t above_c = 0, above_f = 0;
  const int c = warp_suffix_find64(coarse, static_cast<uint32_t>(k), &above_c);
  if (c < 0) return 0u;
  const int f = warp_suffix_find64(fine + c * 64, static_cast<uint32_t>(k) - above_c, &above_f);
  return static_cast<uint32_t>(c * 64 + (f < 0 ? 0 : f));
}

__global__ void __launch_bounds__(NT) topk_hist_build_kernel(const float* scores, int64_t ld, const int32_t* n_valid,
                                                             int64_t n_cols, uint32_t* hist, int chunk) {
  __shared__ uint32_t h[kFine];
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < kFine; i += NT) h[i] = 0u;
  __syncthreads();
  const int64_t row = blockIdx.y;
  const int64_t nv = row_valid(n_valid, row, n_cols);
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  for (int64_t s = c0 + threadIdx.x; s < c1; s += NT) atomicAdd(&h[f2key(scores[row * ld + s]) >> 20], 1u);
  __syncthreads();
  uint32_t* rh = hist + row * kRowWords;
  for (int i = threadIdx.x; i < kFine; i += NT)
    if (h[i]) atomicAdd(&rh[i], h[i]);
  if (threadIdx.x < kCoarse) {
    uint32_t s = 0;
    for (int j = 0; j < 64; ++j) s += h[threadIdx.x * 64 + j];
    if (s) atomicAdd(&rh[kFine + threadIdx.x], s);
  }
}

__global__ void __launch_bounds__(NT) topk_filter_kernel(const float* scores, int64_t ld, const int32_t* n_valid,
                                                         int64_t n_cols, const uint32_t* hist, int k, uint32_t* cnt,
                                                         uint32_t* ckey, int32_t* cpos, int cap, int chunk) {
  __shared__ uint32_t s_b1;
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.y;
  if (threadIdx.x < 32) {
    const uint32_t b1 = threshold_digit(hist + row * kRowWords, k);
    if (threadIdx.x == 0) s_b1 = b1;
  }
  __syncthreads();
  const uint32_t b1 = s_b1;
  const int64_t nv = row_valid(n_valid, row, n_cols);
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  const int lane = threadIdx.x & 31;
  for (int64_t base = c0; base < c1; base += NT) {
    const int64_t s = base + threadIdx.x;
    uint32_t key = 0u;
    if (s < c1) {
      key = f2key(scores[row * ld + s]);
      if (key == 0u) key = 1u;
    }
    const bool take = s < c1 && (key >> 20) >= b1;
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    if (m == 0u) continue;
    uint32_t slot0 = 0;
    if (lane == __ffs(m) - 1) slot0 = atomicAdd(&cnt[row], static_cast<uint32_t>(__popc(m)));
    slot0 = __shfl_sync(0xffffffffu, slot0, __ffs(m) - 1);
    if (take) {
      const uint32_t slot = slot0 + __popc(m & lanemask_lt());
      if (slot < static_cast<uint32_t>(cap)) {
        ckey[row * cap + slot] = key;
        cpos[row * cap + slot] = static_cast<int32_t>(s);
      }
    }
  }
}

// Items are (key, position) pairs: the candidate list in shared memory, or, on overflow, the
// score row itself in position order.
struct FinalItems {
  const uint32_t* key;
  const int32_t* pos;
  const float* row;
  int n;
  bool from_row;
  __device__ __forceinline__ uint32_t k_at(int e) const {
    if (!from_row) return key[e];
    const uint32_t x = f2key(row[e]);
    return x == 0u ? 1u : x;
  }
  __device__ __forceinline__ int32_t p_at(int e) const { return from_row ? e : pos[e]; }
};

__global__ void __launch_bounds__(NT) topk_final_kernel(const float* scores, int64_t ld, const int32_t* n_valid,
                                                        int64_t n_cols, const uint32_t* cnt, const uint32_t* ckey,
                                                        const int32_t* cpos, int cap, int k, int32_t* idx) {
  extern __shared__ uint32_t sm[];
  uint32_t* skey = sm;                                   // [cap]
  int32_t* spos = reinterpret_cast<int32_t*>(sm + cap);  // [cap]
  uint32_t* hist = sm + 2 * cap;                         // [2048] radix / [1024] sort buckets
  uint32_t* tmp = hist + kRadixBins;                     // [32]
  uint32_t* s_res = tmp + 32;                            // [8]
  int32_t* sel = reinterpret_cast<int32_t*>(s_res + 8);  // [k]  winners (unordered)
  int32_t* srt = sel + k;                                // [k]  winners grouped by bucket
  int32_t* eqp = srt + k;                                // [cap] positions of keys equal to T
  const int tid = threadIdx.x, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const int64_t nvr = row_valid(n_valid, row, n_cols);
  const uint32_t n_cand = cnt[row];
  FinalItems it;
  it.from_row = n_cand > static_cast<uint32_t>(cap);
  it.n = it.from_row ? static_cast<int>(nvr) : static_cast<int>(n_cand);
  it.row = scores + row * ld;
  it.key = skey;
  it.pos = spos;
  if (!it.from_row) {
    for (int e = tid; e < it.n; e += NT) {
      skey[e] = ckey[row * cap + e];
      spos[e] = cpos[row * cap + e];
    }
  }
  __syncthreads();

  // ---- exact k-th key: three radix passes (11/11/10 bits)
  uint32_t T = 1u;
  int quota = 0x7fffffff;
  if (it.n > k) {
    uint32_t prefix = 0u, mask = 0u;
    int kk = k;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = shifts[pass], nb = 1 << widths[pass];
      for (int i = tid; i < nb; i += NT) hist[i] = 0u;
      __syncthreads();
      for (int base = 0; base < it.n; base += NT) {
        const int e = base + tid;
        const uint32_t key = e < it.n ? it.k_at(e) : 0u;
        const bool part = key != 0u && (key & mask) == prefix;
        const uint32_t digit = part ? ((key >> shift) & static_cast<uint32_t>(nb - 1)) : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (part && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
      }
      __syncthreads();
      const int bpt = nb / NT;
      const int b0 = tid * bpt;
      uint32_t local = 0;
      for (int q = 0; q < bpt; ++q) local += hist[b0 + q];
      uint32_t tot;
      const uint32_t excl = block_exclusive_scan<NT>(local, tmp, &tot);
      uint32_t run = tot - excl - local;
      for (int q = bpt - 1; q >= 0; --q) {
        const uint32_t h = hist[b0 + q];
        if (run < static_cast<uint32_t>(kk) && run + h >= static_cast<uint32_t>(kk)) {
          s_res[0] = static_cast<uint32_t>(b0 + q);
          s_res[1] = run;
        }
        run += h;
      }
      __syncthreads();
      kk -= static_cast<int>(s_res[1]);
      prefix |= s_res[0] << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      __syncthreads();
    }
    T = prefix;
    quota = kk;
  }

  // ---- winners: every key > T, then the lowest positions among keys == T
  if (tid == 0) {
    s_res[2] = 0u;
    s_res[3] = 0u;
  }
  __syncthreads();
  for (int e = tid; e < it.n; e += NT) {
    const uint32_t key = it.k_at(e);
    if (key == 0u) continue;
    if (key > T) {
      sel[atomicAdd(&s_res[2], 1u)] = it.p_at(e);
    } else if (key == T && !it.from_row) {
      eqp[atomicAdd(&s_res[3], 1u)] = it.p_at(e);
    }
  }
  __syncthreads();
  const int n_gt = static_cast<int>(s_res[2]);
  int take_eq;
  if (!it.from_row) {
    const int n_eq = static_cast<int>(s_res[3]);
    take_eq = min(n_eq, max(0, min(quota, k - n_gt)));
    if (take_eq == n_eq) {
      for (int j = tid; j < n_eq; j += NT) sel[n_gt + j] = eqp[j];
    } else {  // rank the tied positions by counting (ties at the threshold are few)
      for (int j = tid; j < n_eq; j += NT) {
        const int32_t p = eqp[j];
        int rank = 0;
        for (int i = 0; i < n_eq; ++i) rank += eqp[i] < p;
        if (rank < take_eq) sel[n_gt + rank] = p;
      }
    }
  } else {
    // the row is in position order: the first equal keys win
    const int seg = (it.n + NT - 1) / NT;
    const int lo = tid * seg, hi = min(it.n, lo + seg);
    uint32_t c = 0;
    for (int e = lo; e < hi; ++e) c += it.k_at(e) == T;
    uint32_t n_eq;
    uint32_t r = block_exclusive_scan<NT>(c, tmp, &n_eq);
    take_eq = min(static_cast<int>(n_eq), max(0, min(quota, k - n_gt)));
    for (int e = lo; e < hi; ++e)
      if (it.k_at(e) == T) {
        if (r < static_cast<uint32_t>(take_eq)) sel[n_gt + r] = e;
        ++r;
      }
  }
  __syncthreads();
  const int n_sel = n_gt + take_eq;

  // ---- ascending output: counting sort by position bucket, then rank inside the bucket
  int shift = 0;
  while ((nvr >> shift) >= kSortBuckets) ++shift;
  for (int i = tid; i < kSortBuckets; i += NT) hist[i] = 0u;
  __syncthreads();
  for (int j = tid; j < n_sel; j += NT) atomicAdd(&hist[sel[j] >> shift], 1u);
  __syncthreads();
  constexpr int bpt = kSortBuckets / NT;  // 2
  const uint32_t c0 = hist[tid * bpt], c1 = hist[tid * bpt + 1];
  uint32_t tot;
  const uint32_t start = block_exclusive_scan<NT>(c0 + c1, tmp, &tot);
  hist[tid * bpt] = start;  // bucket starts (exclusive prefix)
  hist[tid * bpt + 1] = start + c0;
  __syncthreads();
  uint32_t* fill = hist + kSortBuckets;  // [1024] fill counters (hist has 2048 words)
  for (int i = tid; i < kSortBuckets; i += NT) fill[i] = 0u;
  __syncthreads();
  for (int j = tid; j < n_sel; j += NT) {
    const int32_t p = sel[j];
    const int bkt = p >> shift;
    srt[hist[bkt] + atomicAdd(&fill[bkt], 1u)] = p;
  }
  __syncthreads();
  for (int j = tid; j < n_sel; j += NT) {
    const int32_t p = sel[j];
    const int bkt = p >> shift;
    const int b0 = static_cast<int>(hist[bkt]), n_b = static_cast<int>(fill[bkt]);
    int rank = 0;
    for (int i = 0; i < n_b; ++i) rank += srt[b0 + i] < p;
    idx[row * k + b0 + rank] = p;
  }
  for (int j = n_sel + tid; j < k; j += NT) idx[row * k + j] = -1;
}

struct HistPlan {
  int chunk;
};

HistPlan plan_hist(int64_t rows, int64_t n_cols, int num_sms) {
  HistPlan p{4096};
  while (p.chunk > 1024 && rows * ((n_cols + p.chunk - 1) / p.chunk) < 2 * num_sms) p.chunk /= 2;
  return p;
}

}  // namespace

int topk_hist_cap(int k) { return std::max(8192, 2 * k); }

size_t topk_hist_workspace_bytes(int64_t rows, int k) {
  const int cap = topk_hist_cap(k);
  return 2 * align_up(static_cast<size_t>(rows) * cap * 4, 256);
}

size_t topk_hist_final_smem(int k) {
  return (static_cast<size_t>(topk_hist_cap(k)) * 3 + kRadixBins + 40 + 2 * static_cast<size_t>(k)) * 4;
}

cudaError_t launch_topk_hist(const float* scores, int64_t ld, int64_t rows, int64_t n_cols, const int32_t* n_valid,
                             uint32_t* hist_cnt, int k, int32_t* idx, void* ws_cand, int num_sms, cudaStream_t s) {
  const int cap = topk_hist_cap(k);
  uint32_t* cnt = hist_cnt + rows * kRowWords;
  uint8_t* w = static_cast<uint8_t*>(ws_cand);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(w);
  int32_t* cpos = reinterpret_cast<int32_t*>(w + align_up(static_cast<size_t>(rows) * cap * 4, 256));
  const HistPlan pl = plan_hist(rows, n_cols, num_sms);
  dim3 g1(static_cast<unsigned>(std::max<int64_t>(1, (n_cols + pl.chunk - 1) / pl.chunk)), static_cast<unsigned>(rows));
  const uint32_t* chist = hist_cnt;
  cudaError_t e = launch_pdl(topk_filter_kernel, g1, dim3(NT), 0, s, scores, ld, n_valid, n_cols, chist, k, cnt, ckey,
                             cpos, cap, pl.chunk);
  count_launches(1);
  if (e != cudaSuccess) return e;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(topk_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(topk_hist_final_smem(4096)));
    attr = true;
  }
  const uint32_t* ccnt = cnt;
  const uint32_t* cckey = ckey;
  const int32_t* ccpos = cpos;
  e = launch_pdl(topk_final_kernel, dim3(static_cast<unsigned>(rows)), dim3(NT), topk_hist_final_smem(k), s, scores, ld,
                 n_valid, n_cols, ccnt, cckey, ccpos, cap, k, idx);
  count_launches(1);
  return e;
}

bool topk_uses_hist(int64_t rows, int64_t n_cols, bool has_cand) {
  return !has_cand && rows <= 64 && n_cols >= 16384;
}

size_t topk_hist_standalone_bytes(int64_t rows, int k) {
  return align_up(static_cast<size_t>(rows) * (kRowWords + 1) * 4, 256) + topk_hist_workspace_bytes(rows, k);
}

cudaError_t launch_topk_hist_standalone(const TopkArgs& a, cudaStream_t s) {
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  uint32_t* hist_cnt = reinterpret_cast<uint32_t*>(w);
  const size_t hbytes = static_cast<size_t>(a.rows) * (kRowWords + 1) * 4;
  cudaError_t e = cudaMemsetAsync(hist_cnt, 0, hbytes, s);
  if (e != cudaSuccess) return e;
  const int chunk = 8192;
  dim3 g(static_cast<unsigned>((a.n_cols + chunk - 1) / chunk), static_cast<unsigned>(a.rows));
  e = launch_pdl(topk_hist_build_kernel, g, dim3(NT), 0, s, a.scores, a.ld, a.n_valid, a.n_cols, hist_cnt, chunk);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return launch_topk_hist(a.scores, a.ld, a.rows, a.n_cols, a.n_valid, hist_cnt, a.k, a.idx,
                          w + align_up(hbytes, 256), a.num_sms, s);
}

}  // namespace csa
