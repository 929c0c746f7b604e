// Histogram-guided top-k for long rows (csa_topk, csa_indexer_topk, csa_block_pool).
//
// Same contract as the chunked top-k ("DeepSeek V4-Flash: The Cost of Deciding What to
// Read", section "The Lightning Indexer": keep the k best entries; ties go to the lowest
// position; output ascending, -1 padded).
//
// Every visible score of a row is counted in a histogram of its order-preserving key: 4096
// fine bins (key >> 20) and 64 coarse bins (key >> 26).  The threshold digit b1 is the
// largest fine bin whose suffix count reaches k, so every one of the k best scores has digit
// >= b1.
//  * Few long rows: topk_hist_build_kernel fills the histogram, then topk_select_kernel runs
//    one CTA per 4,096-position chunk:
//    each keeps its scores with digit >= b1, in position order, in its slot of the workspace
//    and takes a ticket; the row's last CTA gathers the slots, finds the exact k-th key by
//    radix passes over the low 20 bits of the b1 bin, takes the lowest positions among equal
//    keys, writes the winners ascending and clears the histogram row.  If the slots overflow
//    (a bin full of ties) it selects over the whole row instead, in position order.
//  * Many long rows (the prefill chunk, the block pool): topk_row_kernel, one CTA per row with
//    the histogram in shared memory and the same exact selection; a long row first estimates
//    b1 from a one-in-eight sample and keeps the scores at or above the estimate when they
//    hold the top k and fit the candidate list (exact b1 from their own histogram), else
//    histograms the whole row.
// The decode step runs topk_select_kernel on the histogram its indexer launch fills.
//
// BF16 scores ("FP4, down to the index scores": the index scores rounded to BF16 before the
// selector) run the same kernels (B16 = true) on the 16-bit order-preserving key, widened to
// 32 bits by 16 zero bits: the fine digit is the same 12 bits (sign, exponent, 3 mantissa
// bits), and the exact refinement inside the threshold bin has 4 bits left instead of 20, one
// radix pass instead of two.
#include <algorithm>
#include <type_traits>

#include <cooperative_groups.h>

#include "csa_internal.h"
#include "csa_ptx.cuh"
#include "select_dev.cuh"

namespace csa {
namespace {

namespace cg = cooperative_groups;

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

// Scores of a row as order-preserving 32-bit keys (0 is reserved for "not a candidate": the
// smallest key maps to 1).  fp32: f2key.  BF16: the 16-bit key (-0 as +0) in the upper half.
template <bool B16>
struct ScoreKey {
  using T = typename std::conditional<B16, uint16_t, float>::type;
  static constexpr int kLowBits = B16 ? 4 : 20;  // refinement bits below the 12-bit digit
  __device__ static __forceinline__ uint32_t of(T x) {
    uint32_t y;
    if constexpr (B16) {
      // negative: all 16 bits flipped; positive (and -0, made +0): the sign bit set
      const uint32_t u = x == 0x8000u ? 0u : static_cast<uint32_t>(x);
      y = (u ^ (((u >> 15) * 0x7FFFu) | 0x8000u)) << 16;
    } else {
      y = f2key(x);
    }
    return y == 0u ? 1u : y;
  }
  __device__ static __forceinline__ T load(const T* p) { return __ldcg(p); }
};

// Eight consecutive keys of a row starting at t0 (< n checked per element; 16-byte vector
// loads when aligned).
template <bool B16>
__device__ __forceinline__ void load_keys8(const typename ScoreKey<B16>::T* srow, int64_t t0, int64_t n,
                                           uint32_t (&key)[8]) {
  using K = ScoreKey<B16>;
  if constexpr (B16) {
    if (t0 + 8 <= n && (reinterpret_cast<uintptr_t>(srow + t0) & 15) == 0) {
      const uint4 x = __ldcg(reinterpret_cast<const uint4*>(srow + t0));
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) key[u] = K::of(static_cast<uint16_t>(w[u >> 1] >> (16 * (u & 1))));
      return;
    }
  } else {
    if (t0 + 8 <= n && (reinterpret_cast<uintptr_t>(srow + t0) & 15) == 0) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(srow + t0));
      const float4 y = __ldcg(reinterpret_cast<const float4*>(srow + t0 + 4));
      const float v[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) key[u] = K::of(v[u]);
      return;
    }
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) key[u] = t0 + u < n ? K::of(K::load(srow + t0 + u)) : 1u;
}

// The exact threshold inside digit b1: the `want` largest keys with that digit are every key
// above *T plus *quota keys equal to *T (radix passes on the refinement bits).
template <bool B16, int NTT, typename F>
__device__ __forceinline__ void select_in_bin(F key_at, int n, int want, uint32_t b1, uint32_t* hist, uint32_t* tmp,
                                              uint32_t* res, uint32_t* T, int* quota, int t) {
  if constexpr (B16) {
    uint32_t t16 = 0;
    team_select_largest<NTT>([key_at](int x) { return key_at(x) >> 16; }, n, want, 4, b1 << 4, 0xFFF0u, hist, tmp,
                             res, &t16, quota, t, 0);
    *T = t16 << 16;
  } else {
    team_select_largest<NTT>(key_at, n, want, 20, b1 << 20, 0xFFF00000u, hist, tmp, res, T, quota, t, 0);
  }
}

__device__ __forceinline__ int64_t row_valid(const int32_t* n_valid, int64_t row, int64_t n_cols) {
  if (!n_valid) return n_cols;
  const int64_t v = n_valid[row];
  return v < 0 ? 0 : (v < n_cols ? v : n_cols);
}

// Slots of a candidate row before its first -1 (the map is ascending positions, then -1
// padding), among the first nv: a 32-way search by the whole warp, identical in every lane.
__device__ int64_t warp_cand_prefix(const int32_t* cm, int64_t nv) {
  const int lane = threadIdx.x & 31;
  int64_t lo = 0, hi = nv;  // the first -1 slot (or nv) lies in [lo, hi]
  while (hi > lo) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t p = lo + lane * step;
    const bool neg = p < hi ? __ldg(cm + p) < 0 : true;
    const uint32_t m = __ballot_sync(0xffffffffu, neg);
    if (m == 0u) {
      lo += 31 * step + 1;
    } else {
      const int f = __ffs(m) - 1;
      if (f == 0) {
        hi = lo;
      } else {
        const int64_t pf = lo + f * step;
        lo += (f - 1) * step + 1;
        hi = pf < hi ? pf : hi;
      }
    }
  }
  return lo;
}

template <bool B16>
__global__ void __launch_bounds__(NT) topk_hist_build_kernel(const void* scores_v, int64_t ld, const int32_t* n_valid,
                                                             int64_t n_cols, uint32_t* hist, int chunk,
                                                             const int32_t* cmap) {
  using K = ScoreKey<B16>;
  const typename K::T* scores = static_cast<const typename K::T*>(scores_v);
  __shared__ uint32_t h[kFine];
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < kFine; i += NT) h[i] = 0u;
  __syncthreads();
  const int64_t row = blockIdx.y;
  int64_t nv = row_valid(n_valid, row, n_cols);
  if (cmap) nv = warp_cand_prefix(cmap + row * n_cols, nv);
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t c1 = c0 + chunk < nv ? c0 + chunk : nv;
  for (int64_t s = c0 + threadIdx.x; s < c1; s += NT) atomicAdd(&h[K::of(scores[row * ld + s]) >> 20], 1u);
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

// One CTA per (row, chunk of kSelChunk positions).  Every CTA finds the threshold digit b1
// of its row from the fine histogram (one read of the 4096 bins; every one of the k best
// scores has digit >= b1), keeps the (key, position) of every score of its chunk with digit
// >= b1, compacted in position order, in its own slot of the workspace, and takes a ticket.
// The CTA that takes a row's last ticket reads the slots back in chunk order (so the row's
// candidates are in position order; with at most 64 chunks the counts and each chunk's first
// 4 NT / n_chunks candidates come in one round trip), finds the exact k-th key among the b1 bin by radix
// passes on its low 20 bits, and writes the winners (every key above it, then the lowest
// positions among keys equal to it) with one stable compaction: the output is already
// ascending.  If the candidates exceed kAllCap (a bin full of ties) it selects over the whole
// row instead.  The tickets (one word per row after the histograms) start at zero.
constexpr int kSelChunk = 4096;           // positions per CTA (8 per thread)
constexpr int kSelPer = kSelChunk / NT;
constexpr int kAllCap = 8192;
constexpr int kSlotCap = 1024;         // candidates one chunk may keep (more: whole-row path)
constexpr int kSlotWords = 4 + 2 * kSlotCap;

constexpr int kMaxChunks = 4096;        // n_cols <= 2^24
constexpr int kMaxChunkPer = kMaxChunks / NT;

struct SelSmem {
  uint32_t cpre[kMaxChunks];  // last CTA: first candidate index of every chunk
  uint32_t ccnt[kMaxChunks];  // last CTA: candidates of every chunk
  uint32_t ak[kAllCap];      // last CTA: the row's candidates in position order
  int32_t ap[kAllCap];
  uint32_t hist[2 * kSortBuckets];
  uint32_t tmp[32];
  uint32_t res[8];
  uint32_t b1, last, n_gt, n_eq;
};

// Decode step: the row's threshold (key T, tie cut P) for the attention, then the row counted
// done (one thread; the fence orders the two words before the count).
__device__ __forceinline__ void publish_threshold(const SelHandoff& ho, int64_t row, uint32_t T, uint32_t P) {
  ho.thr[2 * row] = T;
  ho.thr[2 * row + 1] = P;
  __threadfence();
  atomicAdd(ho.done + row, 1u);
}

size_t sel_smem_bytes(int k) { return sizeof(SelSmem) + 2 * static_cast<size_t>(k) * 4 + 16; }

template <bool B16>
__global__ void __launch_bounds__(NT, 2) topk_select_kernel(const void* scores_v, int64_t ld, const int32_t* n_valid,
                                                         int64_t n_cols, uint32_t* hist, int k, int32_t* idx,
                                                         uint32_t* cand, int n_chunks, const int32_t* cmap,
                                                         const SelHandoff ho) {
  using K = ScoreKey<B16>;
  const typename K::T* scores = static_cast<const typename K::T*>(scores_v);
  extern __shared__ __align__(16) uint8_t sel_raw[];
  SelSmem& S = *reinterpret_cast<SelSmem*>(sel_raw);
  int32_t* sel = reinterpret_cast<int32_t*>(sel_raw + sizeof(SelSmem));  // [k] (whole-row path)
  int32_t* srt = sel + k;                                                // [k] (whole-row path)
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.y;
  const int chunk_id = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const typename K::T* srow = scores + row * ld;
  // this CTA's positions: thread t holds c0 + t*kSelPer .. +kSelPer-1 (contiguous, so the
  // compaction below keeps position order); the loads (bounded by the row length, the
  // visible count is applied after) are in flight with those of n_valid and the histogram
  static_assert(kSelPer == 8, "eight keys a thread");
  const int64_t c0 = static_cast<int64_t>(chunk_id) * kSelChunk;
  uint32_t v[kSelPer];
  const int64_t t0 = c0 + tid * kSelPer;
  load_keys8<B16>(srow, t0, n_cols, v);
  int64_t nvr = row_valid(n_valid, row, n_cols);
  if (cmap) nvr = warp_cand_prefix(cmap + row * n_cols, nvr);
  // histogram rows, then the tickets
  const int64_t rows = gridDim.y;
  uint32_t* ticket = hist + rows * kRowWords + row;
  uint32_t* rh = hist + row * kRowWords;
  const uint32_t b1 = team_threshold_digit<NT>(rh, k, S.tmp, S.res, tid, 0);
  uint32_t key[kSelPer];
  uint32_t cnt = 0;
#pragma unroll
  for (int u = 0; u < kSelPer; ++u) {
    const int64_t s = c0 + tid * kSelPer + u;
    const uint32_t x = v[u];
    key[u] = (s < nvr && (x >> 20) >= b1) ? x : 0u;
    cnt += key[u] != 0u;
  }
  uint32_t n_mine;
  uint32_t off = block_exclusive_scan<NT>(cnt, S.tmp, &n_mine);
  // slot of this chunk: [count, 3 pad][keys x kSlotCap][positions x kSlotCap]
  uint32_t* slot = cand + (static_cast<size_t>(row) * n_chunks + chunk_id) * kSlotWords;
  uint32_t* skey = slot + 4;
  uint32_t* spos = skey + kSlotCap;
#pragma unroll
  for (int u = 0; u < kSelPer; ++u) {
    if (key[u] != 0u) {
      if (off < static_cast<uint32_t>(kSlotCap)) {
        skey[off] = key[u];
        spos[off] = static_cast<uint32_t>(c0 + tid * kSelPer + u);
      }
      ++off;
      // decode step: the candidate's cache row starts towards L2 while the row's last CTA
      // selects (the attention gathers the winners right after)
      if (ho.pf_rows)
        bulk_prefetch_l2(ho.pf_rows + (row * ho.pf_seq_rows + c0 + tid * kSelPer + u) * ho.pf_row_bytes,
                         static_cast<uint32_t>(ho.pf_row_bytes));
    }
  }
  if (tid == 0) slot[0] = n_mine;
  // the last CTA of the row to finish selects (the barrier orders the CTA's slot writes
  // before the fence of the thread that takes the ticket)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (ho.chunks) atomicAdd(ho.chunks + row, 1u);  // decode step: this chunk's slot is readable
    S.last = atomicAdd(ticket, 1u) == static_cast<uint32_t>(n_chunks - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!S.last) return;
  bool publish = false;  // decode step: the row's threshold was published before its list
  __threadfence();
  // every CTA of the row has read the histogram: clear it and the ticket for the next use
  for (int i = tid; i < kRowWords; i += NT) rh[i] = 0u;
  if (tid == 0) *ticket = 0u;

  // ---- the row's last CTA: the chunks' candidate counts and their prefix (one block scan)
  const uint32_t* base = cand + static_cast<size_t>(row) * n_chunks * kSlotWords;
  if (tid == 0) {
    S.n_gt = 0u;
    S.n_eq = 0u;
  }
  uint32_t n_all_u;
  bool any_over;
  // at most NT / 4 chunks (tpc >= 4 threads a chunk): each chunk's count and its first
  // 4 tpc candidates come in one round trip (loads past a chunk's count read unused entries of
  // its slot and are dropped)
  int tpc = 1;
  while (tpc * 2 * n_chunks <= NT) tpc *= 2;
  const bool fused = tpc >= 4;
  const int fch = tid / tpc, fq = tid % tpc;
  uint32_t fk[4], fp[4], fcn = 0, fpre = 0;
  if (fused) {
    if (fch < n_chunks) {
      const uint32_t* sl = base + static_cast<size_t>(fch) * kSlotWords;
      fcn = __ldcg(sl);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        fk[u] = __ldcg(sl + 4 + fq + tpc * u);
        fp[u] = __ldcg(sl + 4 + kSlotCap + fq + tpc * u);
      }
    }
    const uint32_t run = block_exclusive_scan<NT>(fq == 0 ? fcn : 0u, S.tmp, &n_all_u);
    if (fq == 0 && fch < n_chunks) S.cpre[fch] = run;
    any_over = __syncthreads_or(fcn > static_cast<uint32_t>(kSlotCap)) != 0;
    if (fch < n_chunks) fpre = S.cpre[fch];
  } else {
    uint32_t my_n = 0;
    bool my_over = false;
    const int cpt = (n_chunks + NT - 1) / NT;  // chunks per thread (contiguous)
    uint32_t cc[kMaxChunkPer];
#pragma unroll
    for (int q = 0; q < kMaxChunkPer; ++q) {
      const int ch = tid * cpt + q;
      cc[q] = (q < cpt && ch < n_chunks) ? __ldcg(base + static_cast<size_t>(ch) * kSlotWords) : 0u;
      my_n += cc[q];
      my_over |= cc[q] > static_cast<uint32_t>(kSlotCap);
    }
    uint32_t run = block_exclusive_scan<NT>(my_n, S.tmp, &n_all_u);
    any_over = __syncthreads_or(my_over) != 0;
#pragma unroll
    for (int q = 0; q < kMaxChunkPer; ++q) {
      const int ch = tid * cpt + q;
      if (q < cpt && ch < n_chunks) {
        S.cpre[ch] = run;
        S.ccnt[ch] = cc[q];
      }
      run += cc[q];
    }
    __syncthreads();
  }
  const int n_all = static_cast<int>(n_all_u);
  int32_t* orow = idx + row * k;
  // with a candidate map (ascending positions) the winners' slots are written as positions
  const int32_t* cm = cmap ? cmap + row * n_cols : nullptr;
  if (n_all <= kAllCap && !any_over) {
    // the candidates, chunk by chunk in position order: tpc threads a chunk, so every load is in
    // flight at once; the keys above the threshold digit are counted on the way
    uint32_t gt = 0;
    if (fused) {
      if (fch < n_chunks) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t j = static_cast<uint32_t>(fq + tpc * u);
          if (j < fcn) {
            S.ak[fpre + j] = fk[u];
            S.ap[fpre + j] = static_cast<int32_t>(fp[u]);
            gt += (fk[u] >> 20) > b1 ? 1u : 0u;
          }
        }
        const uint32_t* sl = base + static_cast<size_t>(fch) * kSlotWords;
        for (uint32_t j = static_cast<uint32_t>(4 * tpc + fq); j < fcn; j += static_cast<uint32_t>(tpc)) {
          const uint32_t key = __ldcg(sl + 4 + j);
          S.ak[fpre + j] = key;
          S.ap[fpre + j] = static_cast<int32_t>(__ldcg(sl + 4 + kSlotCap + j));
          gt += (key >> 20) > b1 ? 1u : 0u;
        }
      }
    } else {
      for (int ch = tid / tpc; ch < n_chunks; ch += NT / tpc) {
        const uint32_t* sl = base + static_cast<size_t>(ch) * kSlotWords;
        const uint32_t c0 = S.cpre[ch], cn = S.ccnt[ch];
        for (uint32_t j = static_cast<uint32_t>(tid % tpc); j < cn; j += static_cast<uint32_t>(tpc)) {
          const uint32_t key = __ldcg(sl + 4 + j);
          S.ak[c0 + j] = key;
          S.ap[c0 + j] = static_cast<int32_t>(__ldcg(sl + 4 + kSlotCap + j));
          gt += (key >> 20) > b1 ? 1u : 0u;
        }
      }
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    if ((tid & 31) == 0 && gt) atomicAdd(&S.n_gt, gt);
    __syncthreads();
    const uint32_t n_gt = S.n_gt;
    const int need = k - static_cast<int>(n_gt);
    uint32_t T = 1u;
    int quota = 0x7fffffff;
    if (n_all - static_cast<int>(n_gt) > need) {
      const uint32_t* ak = S.ak;
      select_in_bin<B16, NT>([ak](int x) { return ak[x]; }, n_all, need, b1, S.hist, S.tmp, S.res, &T, &quota, tid);
    }
    // the winners in position order: every key above T, then the first quota keys equal to T
    const int seg = (n_all + NT - 1) / NT;
    const int lo = tid * seg, hi = min(n_all, lo + seg);
    uint32_t c_tie = 0, c_ge = 0;
    for (int e = lo; e < hi; ++e) {
      const uint32_t key = S.ak[e];
      c_tie += key == T;
      c_ge += key >= T;
    }
    const uint32_t wt = __reduce_add_sync(0xffffffffu, c_tie);
    if ((tid & 31) == 0 && wt) atomicAdd(&S.n_eq, wt);
    __syncthreads();
    // decode step: a row with few candidates publishes its threshold before the list (the
    // attention masks the candidates it gathered with it)
    publish = ho.cand_cap > 0 && n_all <= ho.cand_cap;
    if (publish && tid == 0 && S.n_eq <= static_cast<uint32_t>(quota)) publish_threshold(ho, row, T, 0x7FFFFFFF);
    if (S.n_eq <= static_cast<uint32_t>(quota)) {
      // every key equal to T wins (the usual case: no tie at the threshold is cut)
      uint32_t n_win;
      uint32_t out = block_exclusive_scan<NT>(c_ge, S.tmp, &n_win);
      for (int e = lo; e < hi; ++e)
        if (S.ak[e] >= T && out < static_cast<uint32_t>(k)) {
          orow[out++] = cm ? cm[S.ap[e]] : S.ap[e];
        }
      for (int j = static_cast<int>(n_win) + tid; j < k; j += NT) orow[j] = -1;
    } else {
      // stable compaction over contiguous segments: ties ranked in position order
      if (publish && tid == 0) S.res[5] = 0xFFFFFFFFu;  // (no key equal to T wins: P = -1)
      uint32_t tie_r = block_exclusive_scan<NT>(c_tie, S.tmp, nullptr);
      if (publish) {
        // the tie cut: the position of the last winning key equal to T (ties are in position order)
        if (tie_r < static_cast<uint32_t>(quota) && tie_r + c_tie >= static_cast<uint32_t>(quota)) {
          uint32_t tr = tie_r;
          for (int e = lo; e < hi; ++e)
            if (S.ak[e] == T && ++tr == static_cast<uint32_t>(quota)) S.res[5] = static_cast<uint32_t>(S.ap[e]);
        }
        __syncthreads();
        if (tid == 0) publish_threshold(ho, row, T, S.res[5]);
      }
      uint32_t c_win = 0;
      {
        uint32_t tr = tie_r;
        for (int e = lo; e < hi; ++e) {
          const uint32_t key = S.ak[e];
          if (key > T) {
            ++c_win;
          } else if (key == T) {
            if (tr < static_cast<uint32_t>(quota)) ++c_win;
            ++tr;
          }
        }
      }
      uint32_t n_win;
      uint32_t out = block_exclusive_scan<NT>(c_win, S.tmp, &n_win);
      for (int e = lo; e < hi; ++e) {
        const uint32_t key = S.ak[e];
        bool w = key > T;
        if (key == T) {
          w = tie_r < static_cast<uint32_t>(quota);
          ++tie_r;
        }
        if (w && out < static_cast<uint32_t>(k)) orow[out++] = cm ? cm[S.ap[e]] : S.ap[e];
      }
      for (int j = static_cast<int>(n_win) + tid; j < k; j += NT) orow[j] = -1;
    }
  } else {
    // too many candidates (a bin full of ties, or crowded into one chunk): select over the whole
    // row in position order
    const typename K::T* rowp = srow;
    auto key_at = [rowp](int x) { return K::of(K::load(rowp + x)); };
    const int n = static_cast<int>(nvr);
    uint32_t T = 1u;
    int quota = 0x7fffffff;
    if (n > k) team_select_largest<NT>(key_at, n, k, 32, 0u, 0u, S.hist, S.tmp, S.res, &T, &quota, tid, 0);
    if (tid == 0) S.n_gt = 0u;
    __syncthreads();
    for (int x = tid; x < n; x += NT)
      if (key_at(x) > T) {
        const uint32_t w = atomicAdd(&S.n_gt, 1u);
        if (w < static_cast<uint32_t>(k)) sel[w] = x;
      }
    __syncthreads();
    const int n_above = min(static_cast<int>(S.n_gt), k);
    const int seg = (n + NT - 1) / NT;
    const int lo = tid * seg, hi = min(n, lo + seg);
    uint32_t c = 0;
    for (int x = lo; x < hi; ++x) c += key_at(x) == T;
    uint32_t n_eqT;
    uint32_t r = block_exclusive_scan<NT>(c, S.tmp, &n_eqT);
    const int take = min(static_cast<int>(n_eqT), max(0, min(quota, k - n_above)));
    for (int x = lo; x < hi; ++x)
      if (key_at(x) == T) {
        if (r < static_cast<uint32_t>(take)) sel[n_above + r] = x;
        ++r;
      }
    __syncthreads();
    team_write_sorted<NT>(sel, n_above + take, k, nvr, S.hist, S.tmp, srt, orow, cm, tid, 0);
  }
  // decode step: the row's list is complete; count it done for the attention waiting on it
  // (the barrier orders every thread's writes before the fence), unless its threshold was
  // published (and counted) already
  if (ho.done && !publish) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(ho.done + row, 1u);
    }
  }
}

// ---- one CTA per row (many long rows: the prefill chunk, the block pool)
// The row is histogrammed in shared memory (4096 fine bins of the order-preserving key), the
// threshold bin b1 found, and the row read again (now from L2) appending the (key, position)
// of every score with digit >= b1 in any order (one shared-memory atomic per warp and batch);
// the exact threshold key T then comes from radix passes inside the b1 bin, ties at T are cut
// to the lowest positions by a radix pass on their positions, and the winners are written
// ascending by a counting sort on their positions.
// The candidate list holds CAP entries: 2048 for k <= 512 (four CTAs fit on an SM), else 8192.
constexpr int kRowPer = 8;                 // scores per thread per batch
constexpr int kRowBatch = kRowPer * NT;    // 4096
constexpr int64_t kSampleMinRow = 16384;   // rows at least this long estimate the threshold first

template <int CAP>
struct RowSmem {
  uint32_t hist[kFine];
  uint32_t ak[CAP];
  int32_t ap[CAP];
  uint32_t sort[2 * kSortBuckets];
  uint32_t tmp[32];
  uint32_t res[8];
  uint32_t n_gt, n_app, n_eq, n_win, n_tie;
};

template <int CAP>
size_t row_smem_bytes(int k) { return sizeof(RowSmem<CAP>) + 2 * static_cast<size_t>(k) * 4 + 16; }

static_assert(kRowPer == 8, "eight keys a thread");

template <int CAP, bool B16>
__global__ void __launch_bounds__(NT, CAP <= 2048 ? 4 : 1) topk_row_kernel(const void* scores_v, int64_t ld, const int32_t* n_valid,
                                                      int64_t n_cols, int k, int32_t* idx, const int32_t* cmap) {
  using K = ScoreKey<B16>;
  const typename K::T* scores = static_cast<const typename K::T*>(scores_v);
  extern __shared__ __align__(16) uint8_t row_raw[];
  RowSmem<CAP>& S = *reinterpret_cast<RowSmem<CAP>*>(row_raw);
  int32_t* sel = reinterpret_cast<int32_t*>(row_raw + sizeof(RowSmem<CAP>));  // [k] (whole-row path)
  int32_t* srt = sel + k;
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  for (int i = tid; i < kFine; i += NT) S.hist[i] = 0u;
  pdl_wait();
  pdl_trigger();
  int64_t nvr = row_valid(n_valid, row, n_cols);
  if (cmap) nvr = warp_cand_prefix(cmap + row * n_cols, nvr);
  const typename K::T* srow = scores + row * ld;
  __syncthreads();
  const int lane = tid & 31;
  // pass 2: the candidates (digit >= bmin), appended in any order (each warp reserves its
  // batch's slots with one shared-memory atomic: no block barrier inside the loop); S.n_app
  // counts them all, S.n_gt those above bmin
  auto collect = [&](uint32_t bmin) {
    if (tid == 0) {
      S.n_gt = 0u;
      S.n_app = 0u;
      S.n_eq = 0u;
      S.n_win = 0u;
      S.n_tie = 0u;
    }
    __syncthreads();
    uint32_t my_gt = 0;
    for (int64_t base = 0; base < nvr; base += kRowBatch) {
      uint32_t v[kRowPer];
      const int64_t t0 = base + static_cast<int64_t>(tid) * kRowPer;
      load_keys8<B16>(srow, t0, nvr, v);
      uint32_t c = 0;
#pragma unroll
      for (int u = 0; u < kRowPer; ++u) {
        const bool in = t0 + u < nvr && (v[u] >> 20) >= bmin;
        c += in;
        my_gt += in && (v[u] >> 20) > bmin;
      }
      uint32_t x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const uint32_t wtot = __shfl_sync(0xffffffffu, x, 31);
      uint32_t wbase = 0;
      if (lane == 31 && wtot) wbase = atomicAdd(&S.n_app, wtot);
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      uint32_t off = wbase + x - c;
#pragma unroll
      for (int u = 0; u < kRowPer; ++u) {
        if (t0 + u < nvr && (v[u] >> 20) >= bmin) {
          if (off < static_cast<uint32_t>(CAP)) {
            S.ak[off] = v[u];
            S.ap[off] = static_cast<int32_t>(t0 + u);
          }
          ++off;
        }
      }
    }
    my_gt = __reduce_add_sync(0xffffffffu, my_gt);
    if (lane == 0 && my_gt) atomicAdd(&S.n_gt, my_gt);
    __syncthreads();
  };
  // Long rows first estimate the threshold digit from a sample, the first 8 scores of every
  // 64: the largest digit whose sample suffix reaches 1.5 k (scaled to the sample) + 16.  If
  // the row holds between k and CAP scores at or above that digit, they are the candidates
  // (every score of the top k is among them) and the exact digit b1 of the k-th largest comes
  // from their own histogram; otherwise the whole row's histogram decides, as below.
  uint32_t b1 = 0u;
  uint32_t n_in = 0u;  // candidates with digit >= b1 (the rest of the list lies below b1)
  bool sampled = false;
  const int64_t n_groups = nvr / 64;
  const int64_t n_s = n_groups * 8;
  if (nvr >= kSampleMinRow && 16 * static_cast<int64_t>(k) <= nvr) {
    for (int64_t g0 = 0; g0 < n_groups; g0 += 2 * NT) {
      uint32_t v[kRowPer], w[kRowPer];
      const int64_t ga = g0 + tid, gb = ga + NT;
      if (ga < n_groups) load_keys8<B16>(srow, ga * 64, nvr, v);
      if (gb < n_groups) load_keys8<B16>(srow, gb * 64, nvr, w);
#pragma unroll
      for (int u = 0; u < kRowPer; ++u) {
        if (ga < n_groups) atomicAdd(&S.hist[v[u] >> 20], 1u);
        if (gb < n_groups) atomicAdd(&S.hist[w[u] >> 20], 1u);
      }
    }
    __syncthreads();
    const int k_s = static_cast<int>(min(n_s, (3 * static_cast<int64_t>(k) * n_s) / (2 * nvr) + 16));
    const uint32_t bs = team_threshold_digit_smem<NT>(S.hist, k_s, S.tmp, S.res, tid, 0);
    collect(bs);
    const uint32_t n_app = S.n_app;
    if (n_app >= static_cast<uint32_t>(k) && n_app <= static_cast<uint32_t>(CAP)) {
      for (int i = tid; i < kFine; i += NT) S.hist[i] = 0u;
      __syncthreads();
      for (int e = tid; e < static_cast<int>(n_app); e += NT) atomicAdd(&S.hist[S.ak[e] >> 20], 1u);
      __syncthreads();
      b1 = team_threshold_digit_smem<NT>(S.hist, k, S.tmp, S.res, tid, 0);
      uint32_t c_gt = 0, c_in = 0;
      for (int e = tid; e < static_cast<int>(n_app); e += NT) {
        const uint32_t dg = S.ak[e] >> 20;
        c_gt += dg > b1;
        c_in += dg >= b1;
      }
      c_gt = __reduce_add_sync(0xffffffffu, c_gt);
      c_in = __reduce_add_sync(0xffffffffu, c_in);
      if (tid == 0) {
        S.n_gt = 0u;
        S.n_tie = 0u;
      }
      __syncthreads();
      if (lane == 0 && c_gt) atomicAdd(&S.n_gt, c_gt);
      if (lane == 0 && c_in) atomicAdd(&S.n_tie, c_in);
      __syncthreads();
      n_in = S.n_tie;
      __syncthreads();
      if (tid == 0) S.n_tie = 0u;
      sampled = true;
    } else {
      for (int i = tid; i < kFine; i += NT) S.hist[i] = 0u;
      __syncthreads();
    }
  }
  if (!sampled) {
    // pass 1: the histogram of the visible scores (two batches of loads in flight)
    for (int64_t base = 0; base < nvr; base += 2 * kRowBatch) {
      uint32_t v[kRowPer], w[kRowPer];
      const int64_t t0 = base + static_cast<int64_t>(tid) * kRowPer, t1 = t0 + kRowBatch;
      load_keys8<B16>(srow, t0, nvr, v);
      load_keys8<B16>(srow, t1, nvr, w);
#pragma unroll
      for (int u = 0; u < kRowPer; ++u) {
        if (t0 + u < nvr) atomicAdd(&S.hist[v[u] >> 20], 1u);
        if (t1 + u < nvr) atomicAdd(&S.hist[w[u] >> 20], 1u);
      }
    }
    __syncthreads();
    b1 = team_threshold_digit_smem<NT>(S.hist, k, S.tmp, S.res, tid, 0);
    collect(b1);
    n_in = S.n_app;
  }
  __syncthreads();
  const uint32_t n_all = S.n_app, n_gt = S.n_gt;
  int32_t* orow = idx + row * k;
  // with a candidate map (ascending positions) the winners' slots are written as positions
  const int32_t* cm = cmap ? cmap + row * n_cols : nullptr;
  if (n_all <= static_cast<uint32_t>(CAP)) {
    const int na = static_cast<int>(n_all);
    const int need = k - static_cast<int>(n_gt);
    uint32_t T = b1 << 20;  // the least key of digit b1: with no cut every candidate >= it wins
    int quota = 0x7fffffff;
    if (static_cast<int>(n_in) - static_cast<int>(n_gt) > need) {
      const uint32_t* ak = S.ak;
      select_in_bin<B16, NT>([ak](int x) { return ak[x]; }, na, need, b1, S.sort, S.tmp, S.res, &T, &quota, tid);
    }
    // the keys equal to T: all of them win unless the quota cuts them; then the quota lowest
    // positions among them win
    uint32_t c_eq = 0;
    for (int e = tid; e < na; e += NT) c_eq += S.ak[e] == T;
    c_eq = __reduce_add_sync(0xffffffffu, c_eq);
    if (lane == 0 && c_eq) atomicAdd(&S.n_eq, c_eq);
    __syncthreads();
    const uint32_t n_eq = S.n_eq;
    int32_t pos_cut = 0x7fffffff;  // ties with a position <= pos_cut win
    if (n_eq > static_cast<uint32_t>(quota) && n_eq <= 256u) {
      // few ties (BF16 scores make them common): list their positions, rank each against the
      // list; the tie of rank quota - 1 is the last winner
      uint32_t* tl = S.sort;
      for (int e = tid; e < na; e += NT)
        if (S.ak[e] == T) tl[atomicAdd(&S.n_tie, 1u)] = static_cast<uint32_t>(S.ap[e]);
      __syncthreads();
      for (int i = tid; i < static_cast<int>(n_eq); i += NT) {
        const uint32_t pi = tl[i];
        int r = 0;
        for (int j = 0; j < static_cast<int>(n_eq); ++j) r += tl[j] < pi;
        if (r == quota - 1) S.res[0] = pi;
      }
      __syncthreads();
      pos_cut = static_cast<int32_t>(S.res[0]);
      __syncthreads();  // S.sort and S.res are reused below
    } else if (n_eq > static_cast<uint32_t>(quota)) {
      // many ties: the quota largest values ~pos among them (positions < 2^24 and distinct, so
      // exactly quota of them), by radix passes on the 24 position bits
      const uint32_t* ak = S.ak;
      const int32_t* ap = S.ap;
      const uint32_t Tk = T;
      uint32_t Tp = 0u;
      int qp = 0;
      team_select_largest<NT>(
          [ak, ap, Tk](int x) { return ak[x] == Tk ? (0x80000000u | (~static_cast<uint32_t>(ap[x]) & 0xFFFFFFu)) : 0u; },
          na, quota, 24, 0x80000000u, 0xFF000000u, S.sort, S.tmp, S.res, &Tp, &qp, tid, 0);
      pos_cut = static_cast<int32_t>(~Tp & 0xFFFFFFu);
    }
    // the winners' positions, appended in any order, then written ascending
    for (int e = tid; e < na; e += NT) {
      const uint32_t key = S.ak[e];
      if (key > T || (key == T && S.ap[e] <= pos_cut)) {
        const uint32_t w = atomicAdd(&S.n_win, 1u);
        if (w < static_cast<uint32_t>(k)) sel[w] = S.ap[e];
      }
    }
    __syncthreads();
    const int n_win = min(static_cast<int>(S.n_win), k);
    team_write_sorted<NT>(sel, n_win, k, nvr, S.sort, S.tmp, srt, orow, cm, tid, 0);
  } else {
    // too many candidates (a bin full of ties): select over the whole row in position order
    const typename K::T* rowp = srow;
    auto key_at = [rowp](int x) { return K::of(K::load(rowp + x)); };
    const int n = static_cast<int>(nvr);
    uint32_t T = 1u;
    int quota = 0x7fffffff;
    if (n > k) team_select_largest<NT>(key_at, n, k, 32, 0u, 0u, S.sort, S.tmp, S.res, &T, &quota, tid, 0);
    if (tid == 0) S.n_gt = 0u;
    __syncthreads();
    for (int x = tid; x < n; x += NT)
      if (key_at(x) > T) {
        const uint32_t w = atomicAdd(&S.n_gt, 1u);
        if (w < static_cast<uint32_t>(k)) sel[w] = x;
      }
    __syncthreads();
    const int n_above = min(static_cast<int>(S.n_gt), k);
    const int seg = (n + NT - 1) / NT;
    const int lo = tid * seg, hi = min(n, lo + seg);
    uint32_t c = 0;
    for (int x = lo; x < hi; ++x) c += key_at(x) == T;
    uint32_t n_eqT;
    uint32_t r = block_exclusive_scan<NT>(c, S.tmp, &n_eqT);
    const int take = min(static_cast<int>(n_eqT), max(0, min(quota, k - n_above)));
    for (int x = lo; x < hi; ++x)
      if (key_at(x) == T) {
        if (r < static_cast<uint32_t>(take)) sel[n_above + r] = x;
        ++r;
      }
    __syncthreads();
    team_write_sorted<NT>(sel, n_above + take, k, nvr, S.sort, S.tmp, srt, orow, cm, tid, 0);
  }
}

}  // namespace

int topk_hist_cap(int k) { return std::max(kAllCap, k); }

int sel_chunks(int64_t n_cols) { return static_cast<int>((n_cols + kSelChunk - 1) / kSelChunk); }
int sel_slot_words() { return kSlotWords; }
int sel_slot_cap() { return kSlotCap; }

// Per-chunk candidate slots ([count, keys, positions] per chunk of every row).
size_t topk_hist_workspace_bytes(int64_t rows, int64_t n_cols) {
  return align_up(static_cast<size_t>(rows) * sel_chunks(n_cols) * kSlotWords * 4, 256);
}

cudaError_t launch_topk_hist(const void* scores, int64_t ld, int64_t rows, int64_t n_cols, const int32_t* n_valid,
                             uint32_t* hist_cnt, int k, int32_t* idx, void* ws_cand, int, cudaStream_t s,
                             const int32_t* cmap, bool bf16, const SelHandoff& ho) {
  static std::atomic<unsigned long long> attr{0};
  if (first_use_in_context(attr)) {
    cudaFuncSetAttribute(topk_select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(sel_smem_bytes(4096)));
    cudaFuncSetAttribute(topk_select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(sel_smem_bytes(4096)));
  }
  const int n_chunks = std::max(1, sel_chunks(n_cols));
  const dim3 grid(static_cast<unsigned>(n_chunks), static_cast<unsigned>(rows));
  const cudaError_t e =
      bf16 ? launch_pdl(topk_select_kernel<true>, grid, dim3(NT), sel_smem_bytes(k), s, scores, ld, n_valid, n_cols,
                        hist_cnt, k, idx, static_cast<uint32_t*>(ws_cand), n_chunks, cmap, ho)
           : launch_pdl(topk_select_kernel<false>, grid, dim3(NT), sel_smem_bytes(k), s, scores, ld, n_valid, n_cols,
                        hist_cnt, k, idx, static_cast<uint32_t*>(ws_cand), n_chunks, cmap, ho);
  count_launches(1);
  return e;
}

// (candidate maps are ascending, so slot order is position order on both paths)
bool topk_uses_hist(int64_t rows, int64_t n_cols, bool) { return rows <= 64 && n_cols >= 16384; }

bool topk_uses_rows(int64_t rows, int64_t n_cols, bool has_cand, int k) {
  return n_cols >= 2048 && k <= 4096 && !topk_uses_hist(rows, n_cols, has_cand);
}

cudaError_t launch_topk_rows(const void* scores, int64_t ld, int64_t rows, int64_t n_cols, const int32_t* n_valid,
                             int k, int32_t* idx, cudaStream_t s, const int32_t* cmap, bool bf16) {
  static std::atomic<unsigned long long> attr{0};
  if (first_use_in_context(attr)) {
    cudaFuncSetAttribute(topk_row_kernel<2048, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(row_smem_bytes<2048>(512)));
    cudaFuncSetAttribute(topk_row_kernel<8192, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(row_smem_bytes<8192>(4096)));
    cudaFuncSetAttribute(topk_row_kernel<2048, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(row_smem_bytes<2048>(512)));
    cudaFuncSetAttribute(topk_row_kernel<8192, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(row_smem_bytes<8192>(4096)));
  }
  const dim3 grid(static_cast<unsigned>(rows));
  cudaError_t e;
  if (k <= 512)
    e = bf16 ? launch_pdl(topk_row_kernel<2048, true>, grid, dim3(NT), row_smem_bytes<2048>(k), s, scores, ld, n_valid,
                          n_cols, k, idx, cmap)
             : launch_pdl(topk_row_kernel<2048, false>, grid, dim3(NT), row_smem_bytes<2048>(k), s, scores, ld,
                          n_valid, n_cols, k, idx, cmap);
  else
    e = bf16 ? launch_pdl(topk_row_kernel<8192, true>, grid, dim3(NT), row_smem_bytes<8192>(k), s, scores, ld, n_valid,
                          n_cols, k, idx, cmap)
             : launch_pdl(topk_row_kernel<8192, false>, grid, dim3(NT), row_smem_bytes<8192>(k), s, scores, ld,
                          n_valid, n_cols, k, idx, cmap);
  count_launches(1);
  return e;
}

size_t topk_hist_standalone_bytes(int64_t rows, int64_t n_cols) {
  return align_up(static_cast<size_t>(rows) * (kRowWords + 1) * 4, 256) + topk_hist_workspace_bytes(rows, n_cols);
}

cudaError_t launch_topk_hist_standalone(const TopkArgs& a, cudaStream_t s) {
  uint8_t* w = static_cast<uint8_t*>(a.ws);
  uint32_t* hist_cnt = reinterpret_cast<uint32_t*>(w);
  const size_t hbytes = static_cast<size_t>(a.rows) * (kRowWords + 1) * 4;
  cudaError_t e = cudaMemsetAsync(hist_cnt, 0, hbytes, s);
  if (e != cudaSuccess) return e;
  const int chunk = 8192;
  dim3 g(static_cast<unsigned>((a.n_cols + chunk - 1) / chunk), static_cast<unsigned>(a.rows));
  e = a.bf16 ? launch_pdl(topk_hist_build_kernel<true>, g, dim3(NT), 0, s, a.scores, a.ld, a.n_valid, a.n_cols,
                          hist_cnt, chunk, a.cand)
             : launch_pdl(topk_hist_build_kernel<false>, g, dim3(NT), 0, s, a.scores, a.ld, a.n_valid, a.n_cols,
                          hist_cnt, chunk, a.cand);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return launch_topk_hist(a.scores, a.ld, a.rows, a.n_cols, a.n_valid, hist_cnt, a.k, a.idx,
                          w + align_up(hbytes, 256), a.num_sms, s, a.cand, a.bf16);
}

}  // namespace csa
