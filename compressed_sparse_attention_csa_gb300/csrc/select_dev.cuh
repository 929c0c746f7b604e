// Block-level selection building blocks shared by the top-k kernel and the decode-step
// indexer: exact k-largest selection by radix passes, the histogram threshold digit, and the
// ascending write of the winners.  NT threads (whole warps) take part; `bar` is the barrier
// they share (0: __syncthreads, else a named barrier over exactly NT threads); `t` is the
// caller's index among them (0..NT-1).
#pragma once
#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {

__device__ __forceinline__ uint32_t lanes_below() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <int NT>
__device__ __forceinline__ void team_sync(int bar) {
  if (bar == 0)
    __syncthreads();
  else
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(NT) : "memory");
}

// Exclusive prefix sum over the team (thread order t); *total gets the sum.
template <int NT>
__device__ __forceinline__ uint32_t team_scan(uint32_t v, int t, uint32_t* tmp, uint32_t* total, int bar) {
  static_assert(NT % 32 == 0 && NT <= 1024, "whole warps");
  const int lane = t & 31, warp = t >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  team_sync<NT>(bar);
  if (warp == 0) {
    uint32_t w = lane < NT / 32 ? tmp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) tmp[lane] = w;
  }
  team_sync<NT>(bar);
  const uint32_t off = warp ? tmp[warp - 1] : 0u;
  if (total) *total = tmp[NT / 32 - 1];
  team_sync<NT>(bar);
  return off + x - v;
}

// Largest-`want` selection among values val(e), e < n, whose bits above `lo_bits` equal
// `prefix` under `mask` (radix passes of up to 10 bits): on return the `want` largest are
// every value > *T plus *quota values equal to *T.  The caller guarantees at least `want`
// values match.  hist: >= 1024 words; res: >= 2 words.
template <int NT, typename F>
__device__ void team_select_largest(F val, int n, int want, int lo_bits, uint32_t prefix, uint32_t mask, uint32_t* hist,
                                    uint32_t* tmp, uint32_t* res, uint32_t* T, int* quota, int t, int bar) {
  int kk = want;
  int shift = lo_bits;
  while (shift > 0) {
    const int wbits = shift < 10 ? shift : 10;
    shift -= wbits;
    const int nb = 1 << wbits;
    for (int i = t; i < nb; i += NT) hist[i] = 0u;
    team_sync<NT>(bar);
    // values of a warp that share a bin are counted with one atomic (the top values of a row
    // often share their leading digits)
    for (int e0 = 0; e0 < n; e0 += NT) {
      const int e = e0 + t;
      const uint32_t v = e < n ? val(e) : 0u;
      const bool in = e < n && (v & mask) == prefix;
      const uint32_t bin = in ? (v >> shift) & static_cast<uint32_t>(nb - 1) : 0xFFFFFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (in && (t & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
    }
    team_sync<NT>(bar);
    // thread t owns `per` consecutive bins counted from the top
    constexpr int per = (1024 + NT - 1) / NT;
    uint32_t local = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      const int bin = nb - 1 - (t * per + q);
      if (bin >= 0) local += hist[bin];
    }
    uint32_t run = team_scan<NT>(local, t, tmp, nullptr, bar);
#pragma unroll
    for (int q = 0; q < per; ++q) {
      const int bin = nb - 1 - (t * per + q);
      if (bin < 0) break;
      const uint32_t h = hist[bin];
      if (run < static_cast<uint32_t>(kk) && run + h >= static_cast<uint32_t>(kk)) {
        res[0] = static_cast<uint32_t>(bin);
        res[1] = run;
      }
      run += h;
    }
    team_sync<NT>(bar);
    kk -= static_cast<int>(res[1]);
    prefix |= res[0] << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    team_sync<NT>(bar);
  }
  *T = prefix;
  *quota = kk;
}

// Largest fine digit (key >> 20, 4096 bins) whose suffix count reaches k, from one read of a
// row's fine histogram in global memory; 0 when the row has fewer than k scores.
template <int NT>
__device__ uint32_t team_threshold_digit(const uint32_t* fine, int k, uint32_t* tmp, uint32_t* res, int t, int bar) {
  constexpr int per = kTopkHistBins / NT;
  static_assert(per % 4 == 0, "16-byte loads");
  uint32_t c[per];
  uint32_t mine = 0;
  // thread t owns bins 4095 - per*t - q (descending), loaded as per/4 16-byte vectors
  // (fine must be 16-byte aligned)
  const uint4* src = reinterpret_cast<const uint4*>(fine + kTopkHistBins - per * (t + 1));
#pragma unroll
  for (int w = 0; w < per / 4; ++w) {
    const uint4 x = __ldcg(src + w);
    c[per - 1 - 4 * w] = x.x;
    c[per - 2 - 4 * w] = x.y;
    c[per - 3 - 4 * w] = x.z;
    c[per - 4 - 4 * w] = x.w;
  }
#pragma unroll
  for (int q = 0; q < per; ++q) mine += c[q];
  if (t == 0) res[4] = 0u;
  uint32_t run = team_scan<NT>(mine, t, tmp, nullptr, bar);
#pragma unroll
  for (int q = 0; q < per; ++q) {
    if (run < static_cast<uint32_t>(k) && run + c[q] >= static_cast<uint32_t>(k))
      res[4] = static_cast<uint32_t>(kTopkHistBins - 1 - (t * per + q));
    run += c[q];
  }
  team_sync<NT>(bar);
  const uint32_t b1 = res[4];
  team_sync<NT>(bar);
  return b1;
}

// The same threshold digit from a histogram in shared memory (16-byte aligned; read as vectors).
template <int NT>
__device__ uint32_t team_threshold_digit_smem(const uint32_t* fine, int k, uint32_t* tmp, uint32_t* res, int t,
                                              int bar) {
  constexpr int per = kTopkHistBins / NT;
  static_assert(per % 4 == 0, "16-byte reads");
  uint32_t c[per];
  uint32_t mine = 0;
  const uint4* src = reinterpret_cast<const uint4*>(fine + kTopkHistBins - per * (t + 1));
#pragma unroll
  for (int w = 0; w < per / 4; ++w) {
    const uint4 x = src[w];
    c[per - 1 - 4 * w] = x.x;
    c[per - 2 - 4 * w] = x.y;
    c[per - 3 - 4 * w] = x.z;
    c[per - 4 - 4 * w] = x.w;
  }
#pragma unroll
  for (int q = 0; q < per; ++q) mine += c[q];
  if (t == 0) res[4] = 0u;
  uint32_t run = team_scan<NT>(mine, t, tmp, nullptr, bar);
#pragma unroll
  for (int q = 0; q < per; ++q) {
    if (run < static_cast<uint32_t>(k) && run + c[q] >= static_cast<uint32_t>(k))
      res[4] = static_cast<uint32_t>(kTopkHistBins - 1 - (t * per + q));
    run += c[q];
  }
  team_sync<NT>(bar);
  const uint32_t b1 = res[4];
  team_sync<NT>(bar);
  return b1;
}

// Winners (distinct positions < nvr) written in ascending position: counting sort by
// position bucket, then rank inside the bucket; -1 after the n_sel winners.  With `map`
// (ascending), winner p is written as map[p].
// hist: >= 2048 words; srt: >= n_sel words.
template <int NT>
__device__ void team_write_sorted(const int32_t* sel, int n_sel, int k, int64_t nvr, uint32_t* hist, uint32_t* tmp,
                                  int32_t* srt, int32_t* out, const int32_t* map, int t, int bar) {
  constexpr int kBuckets = 1024;
  constexpr int per = kBuckets / NT;
  int shift = 0;
  while ((nvr >> shift) >= kBuckets) ++shift;
  for (int i = t; i < kBuckets; i += NT) hist[i] = 0u;
  team_sync<NT>(bar);
  for (int j = t; j < n_sel; j += NT) atomicAdd(&hist[sel[j] >> shift], 1u);
  team_sync<NT>(bar);
  uint32_t c[per];
  uint32_t mine = 0;
#pragma unroll
  for (int q = 0; q < per; ++q) {
    c[q] = hist[t * per + q];
    mine += c[q];
  }
  uint32_t start = team_scan<NT>(mine, t, tmp, nullptr, bar);
#pragma unroll
  for (int q = 0; q < per; ++q) {  // bucket starts (exclusive prefix)
    hist[t * per + q] = start;
    start += c[q];
  }
  uint32_t* fill = hist + kBuckets;
  for (int i = t; i < kBuckets; i += NT) fill[i] = 0u;
  team_sync<NT>(bar);
  for (int j = t; j < n_sel; j += NT) {
    const int32_t p = sel[j];
    const int bkt = p >> shift;
    srt[hist[bkt] + atomicAdd(&fill[bkt], 1u)] = p;
  }
  team_sync<NT>(bar);
  for (int j = t; j < n_sel; j += NT) {
    const int32_t p = sel[j];
    const int bkt = p >> shift;
    const int b0 = static_cast<int>(hist[bkt]), n_b = static_cast<int>(fill[bkt]);
    int rank = 0;
    for (int i = 0; i < n_b; ++i) rank += srt[b0 + i] < p;
    out[b0 + rank] = map ? map[p] : p;
  }
  for (int j = n_sel + t; j < k; j += NT) out[j] = -1;
}

}  // namespace csa
