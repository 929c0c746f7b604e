// Core sparse MQA attention over the selected compressed entries plus the sliding window,
// with a per-head attention sink.
//
// "DeepSeek V4-Flash: The Cost of Deciding What to Read":
//  * "Key and value are the same vector": one cached 512-dim row per entry serves as key and
//    value for all 64 query heads (multi-query);
//  * "Attention sink, and heads that abstain": exp(z'_h) joins the softmax denominator only;
//  * "The sliding window is not an optimisation": the W most recent uncompressed rows are
//    concatenated with the selected entries before the softmax.
// Window rows are positions [max(0, t-W+1), t] that the caller's local rows hold.
//
// Tensor-core path (bf16, d = 512, H = 64).  The rows of one query are gathered 128 at a
// time into shared memory (16-byte cp.async, 128B-swizzled).  The same tile is the A operand
// of both products, K-major for S^T = R Q^T (M = 128 rows, N = 64 heads, K = 512) and
// MN-major for O^T += R^T P^T (M = 128 dims per chunk, N = 64 heads, K = 128 rows), so each
// TMEM lane of S^T is one row and each TMEM lane of O^T one output dim.  The softmax is
// online across row blocks; the row max and row sum over the 128 lanes use a butterfly
// that halves the live values at every step.  The running max is only moved when it grows
// by more than 2^8 (rescaling O^T in TMEM then), which keeps every exponent bounded.
// Decode splits the rows of one query over CTAs and merges the partial (m, l, O) in fixed
// order with the sink; prefill runs one CTA per query.
#include <algorithm>

#include <cuda_fp4.h>

#include "csa_epi.h"
#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ row list helpers
struct RowList {
  int n_sel, n_win;
  int64_t p_lo;
};

// Compacts the valid entries of idx[0:k) into sel[] (kept order) with a block scan.
template <int NT>
__device__ int compact_idx(const int32_t* idx, int k, int64_t E_cap, int32_t* sel, uint32_t* tmp, int* err) {
  const int per = (k + NT - 1) / NT;
  const int lo = threadIdx.x * per, hi = min(k, lo + per);
  uint32_t cnt = 0;
  for (int j = lo; j < hi; ++j) {
    const int32_t v = idx[j];
    if (v >= 0 && v < E_cap) ++cnt;
    else if (v >= E_cap) set_error(err, kErrIndex);
  }
  uint32_t total;
  uint32_t off = block_exclusive_scan<NT>(cnt, tmp, &total);
  for (int j = lo; j < hi; ++j) {
    const int32_t v = idx[j];
    if (v >= 0 && v < E_cap) sel[off++] = v;
  }
  __syncthreads();
  return static_cast<int>(total);
}

// The entry part of a query's row list.  Sparse (CSA): the valid idx entries, compacted into
// sel.  Dense (HCA, "Heavily Compressed Attention": no indexer, every entry it holds): the
// entries s < min(floor((t+1)/m), E_cap), row j being entry j, with no list.
template <int NT>
__device__ int entry_rows(const AttnArgs& a, int64_t r, int64_t t, int32_t* sel, uint32_t* tmp) {
  if (a.dense_m > 0) {
    const int64_t nv = t >= 0 ? (t + 1) / a.dense_m : 0;
    return static_cast<int>(nv < a.E_cap ? nv : a.E_cap);
  }
  return compact_idx<NT>(a.idx + r * a.k, a.k, a.E_cap, sel, tmp, a.err);
}
__device__ __forceinline__ int64_t entry_at(const AttnArgs& a, const int32_t* sel, int j) {
  return a.dense_m > 0 ? j : sel[j];
}

__device__ __forceinline__ void window_of(int64_t t, int W, int64_t base, int64_t L, int64_t& p_lo, int& n_win) {
  int64_t lo = t - W + 1;
  lo = lo > 0 ? lo : 0;
  lo = lo > base ? lo : base;
  int64_t hi = t < base + L - 1 ? t : base + L - 1;
  p_lo = lo;
  n_win = hi >= lo ? static_cast<int>(hi - lo + 1) : 0;
}

// ------------------------------------------------------------------ CUDA-core path
constexpr int kSimtThreads = 256;
constexpr int kSimtTile = 32;

template <typename T>
__global__ void __launch_bounds__(kSimtThreads) attn_simt_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  const int H = a.H, d = a.d, k = a.k;
  float* sq = sm;                           // [H][d]
  float* so = sq + H * d;                   // [H][d]
  float* srow = so + H * d;                 // [32][d+1]
  float* sp = srow + kSimtTile * (d + 1);   // [H][32]
  float* sm_run = sp + H * kSimtTile;       // [H]
  float* sl_run = sm_run + H;
  float* salpha = sl_run + H;
  uint32_t* tmp = reinterpret_cast<uint32_t*>(salpha + H);  // 32
  int32_t* sel = reinterpret_cast<int32_t*>(tmp + 32);      // [k]

  pdl_wait();
  pdl_trigger();
  const int64_t r = blockIdx.x;
  const int b = static_cast<int>(r / a.T);
  const int tid = threadIdx.x;
  const T* q = static_cast<const T*>(a.q) + r * H * d;
  for (int i = tid; i < H * d; i += kSimtThreads) {
    sq[i] = load_f<T>(q + i);
    so[i] = 0.f;
  }
  for (int h = tid; h < H; h += kSimtThreads) {
    sm_run[h] = -INFINITY;
    sl_run[h] = 0.f;
  }
  const int64_t t = a.q_pos[r];
  const int n_sel = entry_rows<kSimtThreads>(a, r, t, sel, tmp);
  int64_t p_lo;
  int n_win;
  window_of(t, a.W, a.local_base[b], a.L, p_lo, n_win);
  const int n_rows = n_sel + n_win;
  const T* kvc = static_cast<const T*>(a.kv_comp) + static_cast<int64_t>(b) * a.E_cap * d;
  const T* kvl = static_cast<const T*>(a.kv_local) + static_cast<int64_t>(b) * a.L * d;
  const int64_t lbase = a.local_base[b];

  for (int r0 = 0; r0 < n_rows; r0 += kSimtTile) {
    const int nr = min(kSimtTile, n_rows - r0);
    for (int i = tid; i < kSimtTile * d; i += kSimtThreads) {
      const int j = i / d, c = i - j * d;
      float v = 0.f;
      if (j < nr) {
        const int lp = r0 + j;
        const T* src = lp < n_sel ? kvc + entry_at(a, sel, lp) * d
                                  : kvl + (p_lo + (lp - n_sel) - lbase) * d;
        v = load_f<T>(src + c);
      }
      srow[j * (d + 1) + c] = v;
    }
    __syncthreads();
    for (int i = tid; i < H * kSimtTile; i += kSimtThreads) {
      const int h = i / kSimtTile, j = i - h * kSimtTile;
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(sq[h * d + c], srow[j * (d + 1) + c], dot);
      sp[i] = j < nr ? dot * a.softmax_scale : -INFINITY;
    }
    __syncthreads();
    for (int h = tid; h < H; h += kSimtThreads) {
      float mx = -INFINITY;
      for (int j = 0; j < nr; ++j) mx = fmaxf(mx, sp[h * kSimtTile + j]);
      const float mold = sm_run[h];
      const float mnew = fmaxf(mold, mx);
      const float alpha = mold == -INFINITY ? 0.f : expf(mold - mnew);
      float sum = 0.f;
      for (int j = 0; j < kSimtTile; ++j) {
        const float e = j < nr ? expf(sp[h * kSimtTile + j] - mnew) : 0.f;
        sp[h * kSimtTile + j] = e;
        sum += e;
      }
      sl_run[h] = sl_run[h] * alpha + sum;
      sm_run[h] = mnew;
      salpha[h] = alpha;
    }
    __syncthreads();
    for (int i = tid; i < H * d; i += kSimtThreads) {
      const int h = i / d, c = i - h * d;
      float acc = so[i] * salpha[h];
      for (int j = 0; j < nr; ++j) acc = fmaf(sp[h * kSimtTile + j], srow[j * (d + 1) + c], acc);
      so[i] = acc;
    }
    __syncthreads();
  }
  T* out = static_cast<T*>(a.out) + r * H * d;
  for (int i = tid; i < H * d; i += kSimtThreads) {
    const int h = i / d;
    const float mr = sm_run[h], sk = a.sink[h];
    const float M = fmaxf(mr, sk);
    const float f = mr == -INFINITY ? 0.f : expf(mr - M);
    const float den = sl_run[h] * f + expf(sk - M);
    store_f<T>(out + i, so[i] * f / den);
  }
  if (a.lse) {
    for (int h = tid; h < H; h += kSimtThreads) {
      const float mr = sm_run[h], sk = a.sink[h];
      const float M = fmaxf(mr, sk);
      const float f = mr == -INFINITY ? 0.f : expf(mr - M);
      a.lse[r * H + h] = M + logf(sl_run[h] * f + expf(sk - M));
    }
  }
}

// ------------------------------------------------------------------ tensor-core path
constexpr int kTcThreads = 256;   // warps 0-3 softmax (S^T lanes), all 8 warps gather / O work
constexpr int kRows = 128;        // rows per block (MMA M of S^T)
constexpr int kD = 512;
constexpr int kH = 64;
constexpr uint32_t kQOff = 0;                       // 8 regions x (64 rows x 128 B)
constexpr uint32_t kROff = kQOff + kH * kD * 2;     // 8 regions x (128 rows x 128 B)
constexpr uint32_t kPOff = kROff + kRows * kD * 2;  // 128 rows x 128 B (MN-major P, N = heads)
constexpr uint32_t kMiscOff = kPOff + kRows * kH * 2;
constexpr int kMaxK = 2048;
constexpr uint32_t kTmemCols = 512;                 // S^T: cols 0..63, O^T: cols 64..319

struct TcAttnSplit {
  int n_split;
  int rows_per_split;
  float* part_o;   // [B*T, n_split, H, d]
  float* part_ml;  // [B*T, n_split, 2, H]
};

// Reduce 64 per-lane values over the 32 lanes of a warp; lane l ends with the results for
// heads 2l and 2l+1 (halving exchange: 32+16+8+4+2 shuffles).
template <bool MAX>
__device__ __forceinline__ float2 warp_reduce64(float (&v)[64]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 32 >> step;  // live values before this step: 2*half
    const int bit = 16 >> step;
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float lo = v[i], hi = v[i + half];
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, bit);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return make_float2(v[0], v[1]);
}
// The same over 32 values; lane l ends with the result for value l.
template <bool MAX>
__device__ __forceinline__ float warp_reduce32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 16 >> step;
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float lo = v[i], hi = v[i + half];
      const float send = upper ? lo : hi;
      const float keep = upper ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const AttnArgs a, const TcAttnSplit sp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kQOff;
  uint8_t* sR = smem + kROff;
  uint8_t* sP = smem + kPOff;
  float* s_mrun = reinterpret_cast<float*>(smem + kMiscOff);  // [64]
  float* s_lrun = s_mrun + kH;
  float* s_mu = s_lrun + kH;
  float* s_alpha = s_mu + kH;
  float* s_red = s_alpha + kH;                                 // [4][64]
  float* s_f = s_red + 4 * kH;                                 // [64]
  uint32_t* tmp = reinterpret_cast<uint32_t*>(s_f + kH);       // [32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(tmp + 32);      // bar_s, bar_o
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + 2);
  int* s_flag = reinterpret_cast<int*>(sTmem + 1);
  int32_t* sel = reinterpret_cast<int32_t*>(s_flag + 4);       // [k]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r = blockIdx.y;
  const int split = blockIdx.x;
  const int b = static_cast<int>(r / a.T);
  const float scale_log2 = a.softmax_scale * kLog2e;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    s_flag[0] = 0;
  }
  if (warp == 4) {
    tmem_alloc(sTmem, kTmemCols);
    tmem_relinquish();
  }
  if (tid < kH) {
    s_mrun[tid] = -INFINITY;
    s_lrun[tid] = 0.f;
  }
  pdl_wait();  // the selection and the caches come from the kernels before this one
  pdl_trigger();
  const int n_sel = compact_idx<kTcThreads>(a.idx + r * a.k, a.k, a.E_cap, sel, tmp, a.err);
  const int64_t t = a.q_pos[r];
  int64_t p_lo;
  int n_win;
  window_of(t, a.W, a.local_base[b], a.L, p_lo, n_win);
  const int n_rows = n_sel + n_win;
  const int row_lo = split * sp.rows_per_split;
  const int row_hi = min(n_rows, row_lo + sp.rows_per_split);
  const int nblk = row_hi > row_lo ? (row_hi - row_lo + kRows - 1) / kRows : 0;

  const __nv_bfloat16* kvc = static_cast<const __nv_bfloat16*>(a.kv_comp) + static_cast<int64_t>(b) * a.E_cap * kD;
  const __nv_bfloat16* kvl = static_cast<const __nv_bfloat16*>(a.kv_local) + static_cast<int64_t>(b) * a.L * kD;
  const int64_t lbase = a.local_base[b];

  // Q: 64 rows x 64 chunks of 16 B
  if (nblk > 0) {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + r * kH * kD;
    for (int i = tid; i < kH * 64; i += kTcThreads) {
      const int h = i >> 6, c = i & 63;
      cp_async16(sQ + (c >> 3) * (kH * 128) + sw128(h, c & 7), q + h * kD + c * 8);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem, tO = tmem + 64;
  const uint32_t qbase = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes

  for (int blk = 0; blk < nblk; ++blk) {
    const int r0 = row_lo + blk * kRows;
    const int nr = min(kRows, row_hi - r0);
    // ---- gather 128 rows x 1 KiB
    for (int i = tid; i < kRows * 64; i += kTcThreads) {
      const int j = i >> 6, c = i & 63;
      uint8_t* dst = sR + (c >> 3) * (kRows * 128) + sw128(j, c & 7);
      if (j < nr) {
        const int lp = r0 + j;
        const __nv_bfloat16* src = lp < n_sel ? kvc + static_cast<int64_t>(sel[lp]) * kD
                                              : kvl + (p_lo + (lp - n_sel) - lbase) * kD;
        cp_async16(dst, src + c * 8);
      } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();

    // ---- S^T = R Q^T
    if (warp == 4 && lane == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kRows, kH, false, false);
      const uint32_t rb = smem_u32(sR), qb = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint32_t reg = ks >> 2, off = (ks & 3) * 32u;
        mma_bf16(tS, smem_desc(rb + reg * (kRows * 128) + off, 16, 1024),
                 smem_desc(qb + reg * (kH * 128) + off, 16, 1024), idesc, ks > 0);
      }
      mma_commit(&bars[0]);
    }
    float x[64];
    if (warp < 4) {
      mbar_wait(&bars[0], blk & 1, a.err, nullptr);
      tc_fence_after();
      float v0[32], v1[32];
      tmem_ld32(tS + qbase, v0);
      tmem_ld32(tS + qbase + 32, v1);
      tmem_wait_ld(v0);
      tmem_wait_ld(v1);
      const bool valid = (warp * 32 + lane) < nr;
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        x[h] = valid ? v0[h] * scale_log2 : -INFINITY;
        x[h + 32] = valid ? v1[h] * scale_log2 : -INFINITY;
      }
      float red[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) red[h] = x[h];
      const float2 mm = warp_reduce64<true>(red);
      s_red[warp * kH + 2 * lane] = mm.x;
      s_red[warp * kH + 2 * lane + 1] = mm.y;
    }
    __syncthreads();
    if (tid < kH) {
      const float mb = fmaxf(fmaxf(s_red[tid], s_red[kH + tid]), fmaxf(s_red[2 * kH + tid], s_red[3 * kH + tid]));
      const float mold = s_mrun[tid];
      float mu = mold;
      if (mold == -INFINITY || mb > mold + 8.f) mu = fmaxf(mold, mb);
      const float alpha = (mu == mold) ? 1.f : exp2f(mold - mu);
      s_mu[tid] = mu;
      s_alpha[tid] = alpha;
      s_mrun[tid] = mu;
      if (alpha != 1.f && blk > 0) s_flag[0] = 1;
    }
    __syncthreads();
    if (warp < 4) {
      const int j = warp * 32 + lane;
      float p[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) {
        const float mu = s_mu[h];
        p[h] = (mu == -INFINITY) ? 0.f : exp2f(x[h] - mu);
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 pk;
        uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 two = __floats2bfloat162_rn(p[c * 8 + 2 * e], p[c * 8 + 2 * e + 1]);
          w[e] = *reinterpret_cast<uint32_t*>(&two);
        }
        *reinterpret_cast<uint4*>(sP + sw128(j, c)) = pk;
      }
      const float2 ss = warp_reduce64<false>(p);
      s_red[warp * kH + 2 * lane] = ss.x;
      s_red[warp * kH + 2 * lane + 1] = ss.y;
      tc_fence_before();
      fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid < kH)
      s_lrun[tid] = s_lrun[tid] * s_alpha[tid] + (s_red[tid] + s_red[kH + tid]) + (s_red[2 * kH + tid] + s_red[3 * kH + tid]);
    if (s_flag[0]) {
      // O^T columns of heads whose reference max moved: scale by alpha
      tc_fence_after();
      const int c_lo = warp < 4 ? 0 : 2;
      for (int cc = c_lo; cc < c_lo + 2; ++cc) {
#pragma unroll
        for (int hc = 0; hc < 64; hc += 32) {
          float v[32];
          const uint32_t ta = tO + qbase + cc * 64 + hc;
          tmem_ld32(ta, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= s_alpha[hc + e];
          tmem_st32(ta, v);
        }
      }
      tmem_wait_st();
      tc_fence_before();
    }
    __syncthreads();
    // ---- O^T += R^T P^T
    if (warp == 4 && lane == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kRows, kH, true, true);
      const uint32_t rb = smem_u32(sR), pb = smem_u32(sP);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int ks = 0; ks < kRows / 16; ++ks) {
          mma_bf16(tO + cc * 64, smem_desc(rb + (2 * cc) * (kRows * 128) + ks * 2048, kRows * 128, 1024),
                   smem_desc(pb + ks * 2048, 8192, 1024), idesc, (blk > 0 || ks > 0) ? 1u : 0u);
        }
      }
      mma_commit(&bars[1]);
    }
    mbar_wait(&bars[1], blk & 1, a.err, nullptr);
    tc_fence_after();
    if (tid == 0) s_flag[0] = 0;
  }

  // ---- epilogue
  const bool single = sp.n_split == 1;
  if (tid < kH) {
    const float mr = s_mrun[tid], lr = s_lrun[tid];
    if (single) {
      const float sk = a.sink[tid] * kLog2e;
      const float M = fmaxf(mr, sk);
      const float f = mr == -INFINITY ? 0.f : exp2f(mr - M);
      const float den = lr * f + exp2f(sk - M);
      s_f[tid] = f / den;
      if (a.lse) a.lse[r * kH + tid] = (M + log2f(den)) * kLn2;
    } else {
      float* ml = sp.part_ml + (r * sp.n_split + split) * 2 * kH;
      ml[tid] = mr;
      ml[kH + tid] = lr;
    }
  }
  __syncthreads();
  if (nblk > 0) {
    const int c_lo = warp < 4 ? 0 : 2;
    for (int cc = c_lo; cc < c_lo + 2; ++cc) {
      const int dd = cc * 128 + (warp & 3) * 32 + lane;
#pragma unroll
      for (int hc = 0; hc < 64; hc += 32) {
        float v[32];
        tmem_ld32(tO + qbase + cc * 64 + hc, v);
        tmem_wait_ld(v);
        if (single) {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + r * kH * kD + dd;
#pragma unroll
          for (int e = 0; e < 32; ++e) o[(hc + e) * kD] = __float2bfloat16_rn(v[e] * s_f[hc + e]);
        } else {
          // partials are stored [dim][head]: this thread's 32 heads are contiguous
          float4* o = reinterpret_cast<float4*>(sp.part_o + ((r * sp.n_split + split) * kD + dd) * kH + hc);
#pragma unroll
          for (int e = 0; e < 32; e += 4) o[e / 4] = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
    }
  } else if (single) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + r * kH * kD;
    for (int i = tid; i < kH * kD; i += kTcThreads) o[i] = __float2bfloat16_rn(0.f);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Fixed-order merge of the split partials with the sink.  One CTA per (row, 4 heads), one
// thread per output dim; partials are [split][dim][head], so each thread reads one float4
// (its 4 heads) per split.
constexpr int kMergeHeads = 4;
constexpr int kMaxSplit = 16;
__global__ void __launch_bounds__(kD) attn_merge_kernel(const AttnArgs a, const TcAttnSplit sp) {
  __shared__ float s_f[kMaxSplit][kMergeHeads];  // per split, per head: 2^(m_s - M) / den
  __shared__ float s_inv[kMergeHeads];
  pdl_wait();
  pdl_trigger();
  const int64_t r = blockIdx.x;
  const int h0 = blockIdx.y * kMergeHeads;
  const int dd = threadIdx.x;
  const int ns = sp.n_split;
  const float* ml = sp.part_ml + r * ns * 2 * kH;
  const float* po = sp.part_o + r * ns * kD * kH;
  if (threadIdx.x < kMergeHeads) {
    const int h = h0 + threadIdx.x;
    const float sk = a.sink[h] * kLog2e;
    float M = sk;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, ml[s * 2 * kH + h]);
    float den = exp2f(sk - M);
    for (int s = 0; s < ns; ++s) {
      const float ms = ml[s * 2 * kH + h];
      const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
      den = fmaf(ml[s * 2 * kH + kH + h], f, den);
      s_f[s][threadIdx.x] = f;
    }
    s_inv[threadIdx.x] = 1.f / den;
    if (a.lse) a.lse[r * kH + h] = (M + log2f(den)) * kLn2;
  }
  __syncthreads();
  float4 o[kMaxSplit];
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s)
    if (s < ns) o[s] = *reinterpret_cast<const float4*>(po + (static_cast<int64_t>(s) * kD + dd) * kH + h0);
  float acc[kMergeHeads] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < kMaxSplit; ++s) {
    if (s < ns && s_f[s][0] + s_f[s][1] + s_f[s][2] + s_f[s][3] > 0.f) {
      acc[0] = fmaf(o[s].x, s_f[s][0], acc[0]);
      acc[1] = fmaf(o[s].y, s_f[s][1], acc[1]);
      acc[2] = fmaf(o[s].z, s_f[s][2], acc[2]);
      acc[3] = fmaf(o[s].w, s_f[s][3], acc[3]);
    }
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (r * kH + h0) * kD + dd;
#pragma unroll
  for (int j = 0; j < kMergeHeads; ++j) out[j * kD] = __float2bfloat16_rn(acc[j] * s_inv[j]);
}

// FP8 main-KV entries: 448 e4m3 codes (28 chunks of 16) then 64 bf16 (8 chunks of 16).
constexpr int kFp8Chunks = (kD - 64) / 16;
constexpr int kFp8RowBytes = (kD - 64) + 64 * 2;
// MXFP4 main-KV entries: 256 payload bytes (E2M1 nibbles) then 32 e4m3 scales (16 dims each).
constexpr int kMxRowBytes = kD / 2 + kD / 16;

// 16 e4m3 codes (one 16-byte load) -> 16 bf16 (exact) as two 16-byte tile chunks
__device__ __forceinline__ void widen_e4m3x16(const uint4& raw, uint4& lo, uint4& hi) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw);
  uint32_t* l = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* h = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2_raw p0 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[e] & 0xFFFFu), __NV_E4M3);
    const __half2_raw p1 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[e] >> 16), __NV_E4M3);
    const __nv_bfloat162 b0 = __float22bfloat162_rn(__half22float2(__half2(p0)));
    const __nv_bfloat162 b1 = __float22bfloat162_rn(__half22float2(__half2(p1)));
    uint32_t* dstw = e < 2 ? l : h;
    dstw[(e & 1) * 2] = *reinterpret_cast<const uint32_t*>(&b0);
    dstw[(e & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&b1);
  }
}
// 8 E2M1 codes (one 32-bit word, element 2i in the low nibble) times their block's e4m3 scale
// -> 8 bf16 (exact: at most 2 + 4 significant bits) as one 16-byte tile chunk
__device__ __forceinline__ uint4 widen_e2m1x8(uint32_t w, uint8_t sc_code) {
  const __half sc = __half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sc_code), __NV_E4M3));
  const __half2 sc2 = __half2half2(sc);
  uint4 o;
  uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2 hh =
        __hmul2(__half2(__nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(w >> (8 * e)), __NV_E2M1)), sc2);
    const __nv_bfloat162 two = __float22bfloat162_rn(__half22float2(hh));
    ow[e] = *reinterpret_cast<const uint32_t*>(&two);
  }
  return o;
}

// ------------------------------------------------------------------ pipelined path (many queries)
// One CTA per query over its whole row list, in tiles of 64 rows that 11 gather warps stage
// (16-byte cp.async, many requests in flight per SM) into two shared-memory buffers while the
// tensor cores and the softmax warps work on the other.
//  * S = Q R^T at M = 64 (heads in TMEM lanes 0-15 of each warp quadrant, the tile's rows in
//    64 columns), into two alternating accumulators, so that S of the next tile overlaps the
//    softmax of this one.  Softmax warp w owns the heads of quadrant w & 3 and rows
//    32 (w >> 2) .. +31 of the tile; the two warps of a quadrant combine their row maxima and
//    sums through shared memory and keep identical running statistics in registers.
//  * O^T += R^T P^T (M = 128 dims a chunk, N = 64 heads, K = 64 rows), P^T K-major: each head
//    thread writes its 32 rows (64 bytes) of the head's 128-byte row.
// Warps 0-7: softmax and output epilogue; warp 8: TMEM owner and MMA issuer; warps 9-19:
// gathers (and the query).
constexpr int kPR = 64;
constexpr int kPfGatherWarps = 11;
constexpr int kPfThreads = 32 * (9 + kPfGatherWarps);
constexpr int kPfMaxK = 2048;
struct PfLayout {
  static constexpr uint32_t kQ = 0;                       // 8 regions x (64 heads x 128 B)
  static constexpr uint32_t kRBytes = kPR * kD * 2;       // one row tile: 8 regions x (64 rows x 128 B)
  static constexpr uint32_t kR = kQ + kH * kD * 2;        // [2] row tiles
  static constexpr uint32_t kPBytes = kH * kPR * 2;       // one P^T tile: 64 heads x 128 B (rows)
  static constexpr uint32_t kP = kR + 2 * kRBytes;        // [2] P^T tiles
  static constexpr uint32_t kMisc = kP + 2 * kPBytes;
  // alpha, f [64] + row-half maxima, sums [2][64] + tmp [32] + flags [4] + barriers [16] + tmem
  static constexpr uint32_t kMiscBytes = (2 * kH + 4 * kH + 32 + 4) * 4 + 16 * 8 + 16;
  static constexpr size_t kSmem = 1024 + kMisc + kMiscBytes + kPfMaxK * 4;
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async16_hint(void* dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "l"(pol)
               : "memory");
}

// KVF: the selected entries' storage: 0 bf16 rows, 1 FP8 entries, 2 MXFP4 entries (widened to
// bf16 in the gather, exactly, so the products are those of the bf16 path over the decoded
// cache); the window rows are bf16 in every case.
template <int KVF>
__global__ void __launch_bounds__(kPfThreads, 1) attn_pf_kernel(const AttnArgs a, const TcAttnSplit sp) {
  using LY = PfLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + LY::kQ;
  uint8_t* sR = smem + LY::kR;
  uint8_t* sP = smem + LY::kP;
  float* s_alpha = reinterpret_cast<float*>(smem + LY::kMisc);  // [64] rescale of the earlier tiles
  float* s_f = s_alpha + kH;                                     // [64] output factor
  float* s_mx = s_f + kH;                                        // [2][64] row-half maxima
  float* s_sm = s_mx + 2 * kH;                                   // [2][64] row-half sums
  uint32_t* tmp = reinterpret_cast<uint32_t*>(s_sm + 2 * kH);    // [32]
  volatile int* s_flag = reinterpret_cast<volatile int*>(tmp + 32);  // [0] rescale, [1] abort
  uint64_t* bars = reinterpret_cast<uint64_t*>(tmp + 32 + 4);    // 8-byte aligned
  uint64_t* full = bars;         // [2] row tile landed (gather threads)
  uint64_t* empty = bars + 2;    // [2] row tile consumed (O^T product committed)
  uint64_t* sfull = bars + 4;    // [2] S accumulator ready
  uint64_t* sempty = bars + 6;   // [2] S accumulator read (softmax threads)
  uint64_t* pfull = bars + 8;    // [2] P^T tile written (softmax threads)
  uint64_t* pempty = bars + 10;  // [2] P^T tile consumed (O^T product committed)
  uint64_t* qfull = bars + 12;   // Q landed (gather threads)
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + 16);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + LY::kMisc + LY::kMiscBytes);  // [k]
  volatile int* sAbort = s_flag + 1;
  constexpr int kSoft = 256, kGath = 32 * kPfGatherWarps;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r = blockIdx.x;
  const int b = static_cast<int>(r / a.T);
  const float scale_log2 = a.softmax_scale * kLog2e;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], kGath);
      mbar_init(&empty[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], kSoft);
      mbar_init(&pfull[i], kSoft);
      mbar_init(&pempty[i], 1);
    }
    mbar_init(qfull, kGath);
    fence_mbar_init();
    s_flag[0] = 0;
    s_flag[1] = 0;
  }
  if (warp == 8) {
    tmem_alloc(sTmem, 512);
    tmem_relinquish();
  }
  pdl_wait();  // the selection and the caches come from the kernels before this one
  pdl_trigger();
  const int64_t t = a.q_pos[r];
  const int n_sel = entry_rows<kPfThreads>(a, r, t, sel, tmp);
  int64_t p_lo;
  int n_win;
  window_of(t, a.W, a.local_base[b], a.L, p_lo, n_win);
  const int n_rows = n_sel + n_win;
  // this CTA's part of the row list (all of it unless the rows are split over CTAs)
  const int split = blockIdx.y;
  const int row_lo = sp.n_split > 1 ? split * sp.rows_per_split : 0;
  const int row_hi = sp.n_split > 1 ? min(n_rows, row_lo + sp.rows_per_split) : n_rows;
  const int nt = row_hi > row_lo ? (row_hi - row_lo + kPR - 1) / kPR : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tO = tmem + 128;  // O^T: 4 chunks x 64 heads; S buffers at columns 0 and 64

  if (warp > 8) {
    // ---- gather warps: thread g copies chunks g, g + 352, ... of the tile (chunk i: row
    //      i / 64, 16-byte piece i % 64); the query likewise
    const int g = tid - 32 * 9;
    const __nv_bfloat16* kvc = static_cast<const __nv_bfloat16*>(a.kv_comp) + static_cast<int64_t>(b) * a.E_cap * kD;
    const uint8_t* kvq = static_cast<const uint8_t*>(a.kv_comp) +
                         static_cast<int64_t>(b) * a.E_cap * (KVF == 1 ? kFp8RowBytes : kMxRowBytes);
    const __nv_bfloat16* kvl = static_cast<const __nv_bfloat16*>(a.kv_local) + static_cast<int64_t>(b) * a.L * kD;
    const int64_t lbase = a.local_base[b];
    // many queries re-read the caches (keep them in L2); a split query reads its rows once
    const uint64_t pol = sp.n_split > 1 ? policy_evict_first() : policy_evict_last();
    if (nt > 0) {
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + r * kH * kD;
      for (int i = g; i < kH * 64; i += kGath) {
        const int h = i >> 6, c = i & 63;
        cp_async16(sQ + (c >> 3) * (kH * 128) + sw128(h, c & 7), q + h * kD + c * 8);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    bool ok = true;
    for (int it = 0; ok && it < nt; ++it) {
      const int buf = it & 1;
      if (it >= 2) {
        if (lane == 0) ok = mbar_wait(&empty[buf], ((it >> 1) & 1) ^ 1, a.err, sAbort);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      uint8_t* dst = sR + buf * LY::kRBytes;
#pragma unroll 4
      for (int i = g; i < kPR * 64; i += kGath) {
        const int j = i >> 6, c = i & 63;
        uint8_t* d = dst + (c >> 3) * (kPR * 128) + sw128(j, c & 7);
        const int lp = row_lo + it * kPR + j;
        if (lp < row_hi) {
          if (KVF != 0 && lp < n_sel) {
            // quantised entry: the FP8 entry's bf16 tail (dims >= d - 64) is copied as is; the
            // rest is widened below
            if (KVF == 1 && c >= kFp8Chunks * 2)
              cp_async16_hint(d, kvq + entry_at(a, sel, lp) * kFp8RowBytes + kFp8Chunks * 16 + (c - kFp8Chunks * 2) * 16,
                              pol);
            continue;
          }
          const __nv_bfloat16* src = lp < n_sel ? kvc + entry_at(a, sel, lp) * kD
                                                : kvl + (p_lo + (lp - n_sel) - lbase) * kD;
          cp_async16_hint(d, src + c * 8, pol);
        } else {
          *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if constexpr (KVF != 0) {
        // the quantised parts of the tile's selected entries: every load of a thread first,
        // then the widening into the swizzled tile (FP8: item = 16 codes -> two chunks;
        // MXFP4: item = 16 payload bytes (32 dims) + their two scale bytes -> four chunks)
        constexpr int kQI = KVF == 1 ? kFp8Chunks : kD / 32;   // items a row
        constexpr int kIt = (kPR * kQI + kGath - 1) / kGath;
        uint4 raw[kIt];
        uint32_t scb[kIt];
#pragma unroll
        for (int u = 0; u < kIt; ++u) {
          const int i = g + u * kGath;
          const int j = i / kQI, q = i - j * kQI;
          const int lp = row_lo + it * kPR + j;
          if (i < kPR * kQI && lp < row_hi && lp < n_sel) {
            const int64_t e = entry_at(a, sel, lp);
            if constexpr (KVF == 1) {
              raw[u] = __ldg(reinterpret_cast<const uint4*>(kvq + e * kFp8RowBytes + q * 16));
            } else {
              raw[u] = __ldg(reinterpret_cast<const uint4*>(kvq + e * kMxRowBytes + q * 16));
              scb[u] = __ldg(reinterpret_cast<const uint16_t*>(kvq + e * kMxRowBytes + kD / 2 + 2 * q));
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kIt; ++u) {
          const int i = g + u * kGath;
          const int j = i / kQI, q = i - j * kQI;
          const int lp = row_lo + it * kPR + j;
          if (i < kPR * kQI && lp < row_hi && lp < n_sel) {
            if constexpr (KVF == 1) {
              uint4 lo, hi;
              widen_e4m3x16(raw[u], lo, hi);
              *reinterpret_cast<uint4*>(dst + ((2 * q) >> 3) * (kPR * 128) + sw128(j, (2 * q) & 7)) = lo;
              *reinterpret_cast<uint4*>(dst + ((2 * q + 1) >> 3) * (kPR * 128) + sw128(j, (2 * q + 1) & 7)) = hi;
            } else {
              const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw[u]);
#pragma unroll
              for (int t4 = 0; t4 < 4; ++t4) {
                const int c = 4 * q + t4;
                *reinterpret_cast<uint4*>(dst + (c >> 3) * (kPR * 128) + sw128(j, c & 7)) =
                    widen_e2m1x8(w[t4], static_cast<uint8_t>(scb[u] >> (8 * (t4 >> 1))));
              }
            }
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      fence_proxy_async_smem();
      if (it == 0) mbar_arrive(qfull);
      mbar_arrive(&full[buf]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  } else if (warp == 8) {
    // ---- MMA issuer: each product as soon as its inputs are ready (polled without
    //      suspending), O^T += R^T P^T first since it frees a row tile for the gathers.
    //      Descriptors are formed once; every MMA adds a constant to the start-address field
    //      (an issue costs about 50 cycles, so the loops carry no descriptor arithmetic).
    if (lane == 0 && nt > 0) {
      const uint32_t idesc_s = idesc_bf16(kH, kPR, false, false);
      const uint32_t idesc_o = idesc_bf16(128, kH, true, false);
      const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024);
      const uint64_t dr0 = smem_desc(smem_u32(sR), 16, 1024);                 // R as S's B operand
      const uint64_t dv0 = smem_desc(smem_u32(sR), kPR * 128, 1024);          // R^T as O^T's A operand
      const uint64_t dp0 = smem_desc(smem_u32(sP), 16, 1024);                 // P^T as O^T's B operand
      constexpr uint64_t kRStep = LY::kRBytes >> 4, kPStep = LY::kPBytes >> 4;
      bool ok = mbar_wait(qfull, 0, a.err, sAbort);
      int ns = 0, np = 0;  // next S tile, next O^T product
      uint64_t t_last = global_ns();
      while (ok && np < nt) {
        if (np < ns && mbar_test_wait(&pfull[np & 1], (np >> 1) & 1)) {
          const int ub = np & 1;
          tc_fence_after();
          const uint64_t dv = dv0 + ub * kRStep, dp = dp0 + ub * kPStep;
          const uint32_t acc0 = np > 0 ? 1u : 0u;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
            for (int ks = 0; ks < kPR / 16; ++ks)
              mma_bf16(tO + cc * 64, dv + (((2 * cc) * (kPR * 128) + ks * 2048) >> 4), dp + ((ks * 32) >> 4), idesc_o,
                       ks > 0 ? 1u : acc0);
          }
          mma_commit(&empty[ub]);
          mma_commit(&pempty[ub]);
          ++np;
          t_last = global_ns();
        } else if (ns < nt && mbar_test_wait(&full[ns & 1], (ns >> 1) & 1) &&
                   (ns < 2 || mbar_test_wait(&sempty[ns & 1], ((ns >> 1) & 1) ^ 1))) {
          const int buf = ns & 1;
          tc_fence_after();
          const uint64_t dr = dr0 + buf * kRStep;
          const uint32_t ts = tmem + buf * 64;
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (kPR * 128) + (ks & 3) * 32;  // kH == kPR: same for Q
            mma_bf16(ts, dq + (off >> 4), dr + (off >> 4), idesc_s, ks > 0 ? 1u : 0u);
          }
          mma_commit(&sfull[buf]);
          ++ns;
          t_last = global_ns();
        } else if (*sAbort) {
          ok = false;
        } else if (global_ns() - t_last > kWaitBudgetNs) {
          set_error(a.err, kErrTimeout);
          *sAbort = 1;
          ok = false;
        }
      }
    }
  } else {
    // ---- softmax warps 0-7: thread (warp w, lane l < 16) has head h = 16 (w & 3) + l (TMEM
    //      lane 32 (w & 3) + l) and rows 32 (w >> 2) .. +31; lanes 16-31 only take part in
    //      the barriers
    const int qd = warp & 3, ch = warp >> 2;
    const int h = qd * 16 + lane;
    const bool own = lane < 16;
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int it = 0; ok && it < nt; ++it) {
      const int buf = it & 1;
      // (wait outcomes are made uniform over the softmax warps: they share named barriers)
      ok = named_and(1, kSoft, mbar_wait(&sfull[buf], (it >> 1) & 1, a.err, sAbort));
      if (!ok) break;
      tc_fence_after();
      float x[32];
      tmem_ld32(tmem + lane_off + buf * 64 + ch * 32, x);
      tmem_wait_ld(x);
      tc_fence_before();
      mbar_arrive(&sempty[buf]);  // S is in registers: the accumulator may take tile it + 2
      float mh = -INFINITY;
      const int r0 = row_lo + it * kPR + ch * 32;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = (r0 + j < row_hi) ? x[j] * scale_log2 : -INFINITY;
        mh = fmaxf(mh, x[j]);
      }
      if (own) s_mx[ch * kH + h] = mh;
      named_sync(1, kSoft);
      const float mb = own ? fmaxf(s_mx[h], s_mx[kH + h]) : -INFINITY;
      // reference max: moved only when the tile's max exceeds it by more than 2^8
      float mu = m_run;
      if (m_run == -INFINITY || mb > m_run + 8.f) mu = fmaxf(m_run, mb);
      const float alpha = (mu == m_run) ? 1.f : ex2_approx(m_run - mu);
      m_run = mu;
      if (own && ch == 0) {
        s_alpha[h] = alpha;
        if (it > 0 && alpha != 1.f) s_flag[0] = 1;
      }
      // the P^T tile of this buffer was last read by the product of tile it - 2
      ok = named_and(1, kSoft, it < 2 || mbar_wait(&pempty[buf], ((it >> 1) & 1) ^ 1, a.err, sAbort));
      if (!ok) break;
      float ps = 0.f;
      {
        uint8_t* prow = sP + buf * LY::kPBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 pk;
          uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = (mu == -INFINITY) ? 0.f : ex2_approx(x[c * 8 + 2 * e] - mu);
            const float p1 = (mu == -INFINITY) ? 0.f : ex2_approx(x[c * 8 + 2 * e + 1] - mu);
            ps += p0 + p1;
            __nv_bfloat162 two = __floats2bfloat162_rn(p0, p1);
            w[e] = *reinterpret_cast<uint32_t*>(&two);
          }
          if (own) *reinterpret_cast<uint4*>(prow + sw128(h, ch * 4 + c)) = pk;
        }
      }
      if (own) s_sm[ch * kH + h] = ps;
      // earlier tiles' O^T columns of heads whose reference max moved: after the product of
      // tile it - 1, scale by alpha (warp w: dims 32 (w & 3) .. of chunks 2 (w >> 2), +1)
      if (s_flag[0] != 0) {
        ok = named_and(1, kSoft, mbar_wait(&pempty[(it - 1) & 1], ((it - 1) >> 1) & 1, a.err, sAbort));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 2 * ch; cc < 2 * ch + 2; ++cc) {
#pragma unroll 1
          for (int hc = 0; hc < 64; hc += 32) {
            float v[32];
            const uint32_t ta = tO + lane_off + cc * 64 + hc;
            tmem_ld32(ta, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= s_alpha[hc + e];
            tmem_st32(ta, v);
          }
        }
        tmem_wait_st();
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&pfull[buf]);
      named_sync(1, kSoft);  // sums written; every thread has read the flag and s_alpha
      if (own) l_run = l_run * alpha + (s_sm[h] + s_sm[kH + h]);
      if (tid == 0) s_flag[0] = 0;
    }
    // ---- epilogue: the last product into O^T, then O / (l + sink) per head
    if (ok && nt > 0)
      ok = named_and(1, kSoft, mbar_wait(&pempty[(nt - 1) & 1], ((nt - 1) >> 1) & 1, a.err, sAbort));
    tc_fence_after();
    if (sp.n_split > 1) {
      // split partial: running (max, sum) per head and the unnormalised O (fp32,
      // [query][split][head][dim]); attn_merge_wide_kernel adds the sink and normalises
      const int64_t ps = r * sp.n_split + split;
      if (own && ch == 0) {
        const bool any = ok && nt > 0;
        sp.part_ml[ps * 2 * kH + h] = any ? m_run : -INFINITY;
        sp.part_ml[ps * 2 * kH + kH + h] = any ? l_run : 0.f;
      }
      if (ok && nt > 0) {
        float* po = sp.part_o + ps * kH * kD;
        for (int cc = 2 * ch; cc < 2 * ch + 2; ++cc) {
          const int dd = cc * 128 + qd * 32 + lane;
#pragma unroll
          for (int hc = 0; hc < 64; hc += 32) {
            float v[32];
            tmem_ld32(tO + lane_off + cc * 64 + hc, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int e = 0; e < 32; ++e) po[(hc + e) * kD + dd] = v[e];
          }
        }
      }
    } else {
    if (own && ch == 0) {
      const float sk = a.sink[h] * kLog2e;
      const float M = fmaxf(m_run, sk);
      const float f = m_run == -INFINITY ? 0.f : exp2f(m_run - M);
      const float den = l_run * f + exp2f(sk - M);
      s_f[h] = f / den;
      if (a.lse) a.lse[r * kH + h] = (M + log2f(den)) * kLn2;
    }
    named_sync(1, kSoft);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + r * kH * kD;
    if (ok && nt > 0) {
      for (int cc = 2 * ch; cc < 2 * ch + 2; ++cc) {
        const int dd = cc * 128 + qd * 32 + lane;
#pragma unroll
        for (int hc = 0; hc < 64; hc += 32) {
          float v[32];
          tmem_ld32(tO + lane_off + cc * 64 + hc, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[(hc + e) * kD + dd] = __float2bfloat16_rn(v[e] * s_f[hc + e]);
        }
      }
    } else {
      for (int i = tid; i < kH * kD; i += kSoft) o[i] = __float2bfloat16_rn(0.f);
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ decode path
// One query row per sequence, its k + W rows split over CTAs: grid (row split, head group,
// query).  A CTA takes 128 rows of the query's row list and NH of the 64 heads (S^T = R Q^T
// with N = NH; O^T += R^T P^T with the P tile zero beyond NH heads).  The list puts the
// window first: the window rows, like the query, are inputs that no earlier kernel of the
// step writes, so they are gathered before the wait on the top-k; the selected rows follow.
// In the decode step a split waits on its own query's step counters (AttnArgs::sel_done)
// rather than on the whole selection kernel, and with few candidates (AttnArgs::cand_cap)
// works on the selection's candidates before the threshold that picks them is published:
// split 0 the window, split s the candidates 128 (s - 1) .. +127; the softmax keeps a
// candidate iff its key is above the threshold key, or equal to it at a position up to the
// tie cut.  Partials are stored [query][split][head][dim] (each warp store is 128 contiguous
// bytes) and merged, with the sink, by attn_merge_wide_kernel.


template <int NH>
struct DecLayout {
  static constexpr uint32_t kQ = 0;                          // 8 regions x (NH rows x 128 B)
  static constexpr uint32_t kR = kQ + NH * kD * 2;           // 8 regions x (128 rows x 128 B)
  static constexpr uint32_t kP = kR + kRows * kD * 2;        // 128 rows x 128 B (64 head columns)
  static constexpr uint32_t kMisc = kP + kRows * 128;
  static constexpr uint32_t kMiscBytes = (NH * 8 + 32) * 4 + 64;  // m, l, f, red[4], tmp; bars; tmem
  static constexpr size_t kSmem = 1024 + kMisc + kMiscBytes + kMaxK * 4;
};

template <int NH, int KVF>  // KVF: 0 bf16 entries, 1 FP8 entries, 2 MXFP4 entries
__global__ void __launch_bounds__(kTcThreads, 1) attn_dec_kernel(const AttnArgs a, const TcAttnSplit sp) {
  using LY = DecLayout<NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + LY::kQ;
  uint8_t* sR = smem + LY::kR;
  uint8_t* sP = smem + LY::kP;
  float* s_m = reinterpret_cast<float*>(smem + LY::kMisc);  // [NH] block max (log2 units)
  float* s_l = s_m + NH;                                     // [NH] block sum
  float* s_f = s_l + NH;                                     // [NH] output factor
  float* s_red = s_f + NH;                                   // [4][NH]
  uint32_t* tmp = reinterpret_cast<uint32_t*>(s_red + 4 * NH);  // [32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(tmp + 32 + ((NH * 7) & 1));  // 8-byte aligned
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + 2);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + LY::kMisc + LY::kMiscBytes);  // [k]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r = blockIdx.z;
  const int h0 = blockIdx.y * NH;
  const int split = blockIdx.x;
  const int b = static_cast<int>(r / a.T);
  const float scale_log2 = a.softmax_scale * kLog2e;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(sTmem, kTmemCols);
    tmem_relinquish();
  }
  if constexpr (NH < kH) {  // head columns of P beyond this CTA's heads stay zero
    for (int i = tid; i < kRows * 8; i += kTcThreads) {
      const int j = i >> 3, c = i & 7;
      if (c >= NH / 8) *reinterpret_cast<uint4*>(sP + sw128(j, c)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // the query and the window rows: inputs, loaded before the wait
  const int64_t t = a.q_pos[r];
  const int64_t lbase = a.local_base[b];
  int64_t p_lo;
  int n_win;
  window_of(t, a.W, lbase, a.L, p_lo, n_win);
  int row_lo = split * sp.rows_per_split;  // (candidate mode: reset to 0 below)
  const int row_cap = row_lo + kRows;
  const __nv_bfloat16* kvc = static_cast<const __nv_bfloat16*>(a.kv_comp) + static_cast<int64_t>(b) * a.E_cap * kD;
  const __nv_bfloat16* kvl = static_cast<const __nv_bfloat16*>(a.kv_local) + static_cast<int64_t>(b) * a.L * kD;
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q) + (r * kH + h0) * kD;
    for (int i = tid; i < NH * 64; i += kTcThreads) {
      const int h = i >> 6, c = i & 63;
      cp_async16(sQ + (c >> 3) * (NH * 128) + sw128(h, c & 7), q + h * kD + c * 8);
    }
    const int w_hi = min(n_win, row_cap);
    for (int i = tid; i < kRows * 64; i += kTcThreads) {
      const int j = i >> 6, c = i & 63;
      const int lp = row_lo + j;
      if (lp < w_hi) cp_async16(sR + (c >> 3) * (kRows * 128) + sw128(j, c & 7), kvl + (p_lo + lp - lbase) * kD + c * 8);
    }
  }
  int row_hi;
  // candidate mode (decode step, few candidates): split 0 holds the window rows only, split
  // s > 0 the selection's candidates 128 (s - 1) .. +127 (in slot order), gathered before the
  // threshold is known and masked by it in the softmax; skey: their keys
  bool cand = false;
  uint32_t* skey = reinterpret_cast<uint32_t*>(sel + kRows);        // [kRows]
  uint32_t* cpre = skey + kRows;                                     // [64] chunk prefix, then n_all
  bool list_mode = true;
  if (a.sel_done && a.cand_cap > 0) {
    pdl_trigger();
    if (tid == 0) wait_count(a.sel_chunks + r, static_cast<uint32_t>(a.sel_n_chunks), a.err);
    __syncthreads();
    const uint32_t* sb = a.sel_slots + static_cast<size_t>(r) * a.sel_n_chunks * a.sel_slot_words;
    if (warp == 0) {
      // the chunks' candidate counts (at most 64) and their exclusive prefix
      const uint32_t c0 = lane < a.sel_n_chunks ? __ldcg(sb + static_cast<size_t>(lane) * a.sel_slot_words) : 0u;
      const uint32_t c1 =
          lane + 32 < a.sel_n_chunks ? __ldcg(sb + static_cast<size_t>(lane + 32) * a.sel_slot_words) : 0u;
      uint32_t i0 = c0, i1 = c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v0 = __shfl_up_sync(0xffffffffu, i0, o), v1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
          i0 += v0;
          i1 += v1;
        }
      }
      const uint32_t t0 = __shfl_sync(0xffffffffu, i0, 31), t1 = __shfl_sync(0xffffffffu, i1, 31);
      cpre[lane] = i0 - c0;
      cpre[lane + 32] = t0 + i1 - c1;
      if (lane == 0) cpre[64] = t0 + t1;
    }
    __syncthreads();
    const int n_all = static_cast<int>(cpre[64]);
    if (n_all <= a.cand_cap) {
      list_mode = false;
      if (split == 0) {
        row_hi = n_win;  // the window rows, loaded above
      } else {
        cand = true;
        const int g0 = (split - 1) * kRows;
        row_lo = 0;
        n_win = 0;
        row_hi = min(max(n_all - g0, 0), kRows);
        if (tid < row_hi) {
          const int gi = g0 + tid;
          int lo = 0, hi = a.sel_n_chunks - 1;  // the last chunk whose prefix is <= gi
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<int>(cpre[mid]) <= gi) lo = mid;
            else hi = mid - 1;
          }
          const uint32_t* sl = sb + static_cast<size_t>(lo) * a.sel_slot_words;
          const int e = gi - static_cast<int>(cpre[lo]);
          skey[tid] = __ldcg(sl + 4 + e);
          sel[tid] = static_cast<int32_t>(__ldcg(sl + 4 + a.sel_slot_cap + e));
        }
        __syncthreads();
      }
    }
  }
  if (a.sel_done && list_mode) {
    // decode step: wait for this query's list only (counted done by the selection's last CTA
    // of the row once written), not for the whole selection kernel; the list holds its entries
    // first, so this split reads just its own slice, and its valid rows are a prefix
    if (tid == 0) wait_count(a.sel_done + r, __ldcg(a.sel_seen + r) + 1u, a.err);
    __syncthreads();
    pdl_trigger();
    bool valid = false;
    if (tid < kRows) {
      const int lp = row_lo + tid, e = lp - n_win;
      valid = lp < n_win;
      if (e >= 0 && e < a.k) {
        int32_t v = __ldcg(a.idx + r * a.k + e);
        if (v >= a.E_cap) {
          set_error(a.err, kErrIndex);
          v = -1;
        }
        sel[e] = v;
        valid = v >= 0;
      }
    }
    row_hi = row_lo + __syncthreads_count(valid);
  } else if (!a.sel_done) {
    pdl_wait();  // the selection (and the entry compressed this step) come from earlier kernels
    pdl_trigger();
    const int n_sel = compact_idx<kTcThreads>(a.idx + r * a.k, a.k, a.E_cap, sel, tmp, a.err);
    row_hi = min(n_win + n_sel, row_cap);
  }
  const int nr = row_hi - row_lo;  // rows of this split (<= 0: none)
  if constexpr (KVF == 0) {
    // thread = one 16-byte column c of rows j0, j0 + 4, ...: a warp moves 512 contiguous bytes
    // of a row, and the copy's addresses cost an add and a multiply-add
    static_assert(kTcThreads == 256, "four rows a pass");
    const int c = tid & 63, j0 = tid >> 6;
    uint8_t* dcol = sR + (c >> 3) * (kRows * 128);
    const __nv_bfloat16* scol = kvc + c * 8;
#pragma unroll 8
    for (int j = j0; j < kRows; j += 4) {
      const int lp = row_lo + j;
      uint8_t* dst = dcol + sw128(j, c & 7);
      if (lp >= row_hi) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      } else if (lp >= n_win) {
        cp_async16(dst, scol + static_cast<int64_t>(sel[lp - n_win]) * kD);
      }
    }
  } else if constexpr (KVF == 1) {
    // FP8 entries (576 B: e4m3 dims 0..447, bf16 dims 448..511): a row is 36 chunks of 16 B;
    // chunk q < 28 holds dims 16q .. 16q+15 as e4m3 (two bf16 chunks of the tile once
    // converted), chunk q >= 28 bf16 dims 448 + 8 (q - 28) .. (copied as they are).  Every
    // load of a thread is issued before the first conversion.
    constexpr int kQ = kFp8RowBytes / 16, kItems = (kRows * kQ + kTcThreads - 1) / kTcThreads;
    const uint8_t* kvb = static_cast<const uint8_t*>(a.kv_comp) + static_cast<int64_t>(b) * a.E_cap * kFp8RowBytes;
    uint4 raw[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kTcThreads;
      if (i >= kRows * kQ) break;
      const int j = i / kQ, q = i - j * kQ;
      const int lp = row_lo + j;
      if (lp >= row_hi) {
        if (q < kFp8Chunks) {
          *reinterpret_cast<uint4*>(sR + ((2 * q) >> 3) * (kRows * 128) + sw128(j, (2 * q) & 7)) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(sR + ((2 * q + 1) >> 3) * (kRows * 128) + sw128(j, (2 * q + 1) & 7)) =
              make_uint4(0u, 0u, 0u, 0u);
        } else {
          const int c = 2 * kFp8Chunks + (q - kFp8Chunks);
          *reinterpret_cast<uint4*>(sR + (c >> 3) * (kRows * 128) + sw128(j, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
        }
      } else if (lp >= n_win) {
        const uint8_t* src = kvb + static_cast<int64_t>(sel[lp - n_win]) * kFp8RowBytes + q * 16;
        if (q < kFp8Chunks) {
          raw[u] = __ldg(reinterpret_cast<const uint4*>(src));
        } else {
          const int c = 2 * kFp8Chunks + (q - kFp8Chunks);
          cp_async16(sR + (c >> 3) * (kRows * 128) + sw128(j, c & 7), src);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kTcThreads;
      if (i >= kRows * kQ) break;
      const int j = i / kQ, q = i - j * kQ;
      const int lp = row_lo + j;
      if (lp < row_hi && lp >= n_win && q < kFp8Chunks) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw[u]);
        uint4 lo, hi;
        uint32_t* l = reinterpret_cast<uint32_t*>(&lo);
        uint32_t* h = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // 4 e4m3 codes -> 4 bf16
          const __half2_raw p0 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[e] & 0xFFFFu), __NV_E4M3);
          const __half2_raw p1 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[e] >> 16), __NV_E4M3);
          const __nv_bfloat162 b0 = __float22bfloat162_rn(__half22float2(__half2(p0)));
          const __nv_bfloat162 b1 = __float22bfloat162_rn(__half22float2(__half2(p1)));
          uint32_t* dstw = e < 2 ? l : h;
          dstw[(e & 1) * 2] = *reinterpret_cast<const uint32_t*>(&b0);
          dstw[(e & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&b1);
        }
        *reinterpret_cast<uint4*>(sR + ((2 * q) >> 3) * (kRows * 128) + sw128(j, (2 * q) & 7)) = lo;
        *reinterpret_cast<uint4*>(sR + ((2 * q + 1) >> 3) * (kRows * 128) + sw128(j, (2 * q + 1) & 7)) = hi;
      }
    }
  } else {
    // MXFP4 entries (288 B): payload chunk q (16 B) holds dims 32q .. 32q+31 as E2M1 nibbles
    // (element 2i in the low nibble), scale bytes 256 + 2q, 2q+1 (e4m3) cover dims 32q .. +15
    // and 32q+16 .. +31; widened to bf16 (exact: <= 2 + 4 significant bits) into tile chunks
    // 4q .. 4q+3.  Every load of a thread is issued before the first conversion.
    constexpr int kQ = kD / 32, kItems = kRows * kQ / kTcThreads;
    const uint8_t* kvb = static_cast<const uint8_t*>(a.kv_comp) + static_cast<int64_t>(b) * a.E_cap * kMxRowBytes;
    uint4 raw[kItems];
    uint32_t scb[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kTcThreads;
      const int j = i / kQ, q = i - j * kQ;
      const int lp = row_lo + j;
      if (lp >= row_hi) {
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          const int c = 4 * q + t4;
          *reinterpret_cast<uint4*>(sR + (c >> 3) * (kRows * 128) + sw128(j, c & 7)) = make_uint4(0u, 0u, 0u, 0u);
        }
      } else if (lp >= n_win) {
        const uint8_t* src = kvb + static_cast<int64_t>(sel[lp - n_win]) * kMxRowBytes;
        raw[u] = __ldg(reinterpret_cast<const uint4*>(src + 16 * q));
        scb[u] = __ldg(reinterpret_cast<const uint16_t*>(src + kD / 2 + 2 * q));
      }
    }
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      const int i = tid + u * kTcThreads;
      const int j = i / kQ, q = i - j * kQ;
      const int lp = row_lo + j;
      if (lp < row_hi && lp >= n_win) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw[u]);
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {  // 8 dims = one 32-bit word of nibbles
          // E2M1 pairs -> half2 (hardware conversion), times the block's e4m3 scale in half2
          // (exact: at most 2 + 4 significant bits, 2^-10 .. 2688), then bf16 (exact)
          const __half sc = __half(__nv_cvt_fp8_to_halfraw(
              static_cast<__nv_fp8_storage_t>(scb[u] >> (8 * (t4 >> 1))), __NV_E4M3));
          const __half2 sc2 = __half2half2(sc);
          uint4 o;
          uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 h = __hmul2(
                __half2(__nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(w[t4] >> (8 * e)), __NV_E2M1)),
                sc2);
            const __nv_bfloat162 two = __float22bfloat162_rn(__half22float2(h));
            ow[e] = *reinterpret_cast<const uint32_t*>(&two);
          }
          const int c = 4 * q + t4;
          *reinterpret_cast<uint4*>(sR + (c >> 3) * (kRows * 128) + sw128(j, c & 7)) = o;
        }
      }
    }
  }
  cp_async_wait_all();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem, tO = tmem + 64;
  const uint32_t qbase = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes

  if (nr > 0) {
    // ---- S^T = R Q^T  (M = 128 rows, N = NH heads, K = 512)
    if (warp == 4 && lane == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kRows, NH, false, false);
      const uint32_t rb = smem_u32(sR), qb = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint32_t reg = ks >> 2, off = (ks & 3) * 32u;
        mma_bf16(tS, smem_desc(rb + reg * (kRows * 128) + off, 16, 1024),
                 smem_desc(qb + reg * (NH * 128) + off, 16, 1024), idesc, ks > 0);
      }
      mma_commit(&bars[0]);
    }
    // softmax on all 8 warps: warp w takes TMEM lanes 32 (w & 3) .. +31 (a lane is a row) and
    // heads HH (w >> 2) .. +HH-1 of the CTA's NH
    constexpr int HH = NH / 2;
    const int hh0 = (warp >> 2) * HH;
    float x[HH];
    uint32_t thr_t = 0u;  // candidate mode: the published threshold (key, tie cut)
    int32_t thr_p = 0;
    if (cand) {
      if (tid == 0) wait_count(a.sel_done + r, __ldcg(a.sel_seen + r) + 1u, a.err);
      __syncthreads();
      thr_t = __ldcg(a.sel_thr + 2 * r);
      thr_p = static_cast<int32_t>(__ldcg(a.sel_thr + 2 * r + 1));
    }
    {
      mbar_wait(&bars[0], 0, a.err, nullptr);
      tc_fence_after();
      const int jr = (warp & 3) * 32 + lane;
      bool valid = jr < nr;
      if (cand && valid) {
        const uint32_t kj = skey[jr];
        valid = kj > thr_t || (kj == thr_t && sel[jr] <= thr_p);
        if (!valid) {  // a candidate left out: zero this half of its row (P = 0, and 0 x NaN is NaN)
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(sR + ((warp >> 2) * 4 + g) * (kRows * 128) + sw128(jr, c)) =
                  make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float v[32];
      tmem_ld32(tS + qbase + hh0, v);  // (columns past NH are read and ignored)
      tmem_wait_ld(v);
#pragma unroll
      for (int e = 0; e < HH; ++e) x[e] = valid ? v[e] * scale_log2 : -INFINITY;
#pragma unroll
      for (int h = 0; h < HH; ++h) {
        float mx = x[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_red[warp * HH + h] = mx;  // [head half][quadrant][HH]
      }
    }
    __syncthreads();
    {
      const int j = (warp & 3) * 32 + lane;
      const float* rm = s_red + (warp >> 2) * 4 * HH;
      float p[HH];
#pragma unroll
      for (int h = 0; h < HH; ++h) {
        const float mu = fmaxf(fmaxf(rm[h], rm[HH + h]), fmaxf(rm[2 * HH + h], rm[3 * HH + h]));
        p[h] = (mu == -INFINITY) ? 0.f : exp2f(x[h] - mu);
      }
#pragma unroll
      for (int c = 0; c < HH / 8; ++c) {
        uint4 pk;
        uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 two = __floats2bfloat162_rn(p[c * 8 + 2 * e], p[c * 8 + 2 * e + 1]);
          w[e] = *reinterpret_cast<uint32_t*>(&two);
        }
        *reinterpret_cast<uint4*>(sP + sw128(j, hh0 / 8 + c)) = pk;
      }
      float sm[HH];
#pragma unroll
      for (int h = 0; h < HH; ++h) {
        sm[h] = p[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sm[h] += __shfl_xor_sync(0xffffffffu, sm[h], o);
      }
      // (every thread has read s_red's maxima before the sums overwrite the other half)
      if (tid < NH) {
        const float* qm = s_red + (tid / HH) * 4 * HH + tid % HH;
        s_m[tid] = fmaxf(fmaxf(qm[0], qm[HH]), fmaxf(qm[2 * HH], qm[3 * HH]));
      }
      __syncthreads();
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < HH; ++h) s_red[warp * HH + h] = sm[h];
      }
      tc_fence_before();
      fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid < NH) {
      const float* ql = s_red + (tid / HH) * 4 * HH + tid % HH;
      s_l[tid] = (ql[0] + ql[HH]) + (ql[2 * HH] + ql[3 * HH]);
    }
    // ---- O^T = R^T P^T  (M = 128 dims per chunk, N = 64 head columns, K = 128 rows)
    if (warp == 4 && lane == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kRows, kH, true, true);
      const uint32_t rb = smem_u32(sR), pb = smem_u32(sP);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int ks = 0; ks < kRows / 16; ++ks) {
          mma_bf16(tO + cc * 64, smem_desc(rb + (2 * cc) * (kRows * 128) + ks * 2048, kRows * 128, 1024),
                   smem_desc(pb + ks * 2048, 8192, 1024), idesc, ks > 0 ? 1u : 0u);
        }
      }
      mma_commit(&bars[1]);
    }
    mbar_wait(&bars[1], 0, a.err, nullptr);
    tc_fence_after();
  } else if (tid < NH) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  __syncthreads();

  // ---- epilogue: (m, l) and the unnormalised O of this split's heads
  if (tid < NH) {
    float* ml = sp.part_ml + (r * sp.n_split + split) * 2 * kH;
    ml[h0 + tid] = s_m[tid];
    ml[kH + h0 + tid] = s_l[tid];
  }
  const int c_lo = warp < 4 ? 0 : 2;
  for (int cc = c_lo; cc < c_lo + 2; ++cc) {
    const int dd = cc * 128 + (warp & 3) * 32 + lane;
    float* o = sp.part_o + ((r * sp.n_split + split) * kH + h0) * kD + dd;
#pragma unroll
    for (int hc = 0; hc < NH; hc += 32) {
      float v[32];
      if (nr > 0) {
        tmem_ld32(tO + qbase + cc * 64 + hc, v);
        tmem_wait_ld(v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (hc + e < NH) o[(hc + e) * kD] = v[e];
    }
  }
  if (a.sel_done) pdl_wait();  // complete only after the selection: keeps the stream order
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ dense rows, few queries
// HCA decode ("Heavily Compressed Attention": every entry the layer holds, plus the window,
// with the sink).  Grid (split, query): a query's entries are cut into splits of up to
// kHdTiles x 128 rows and its window rows form one more split.  The rows of a split are
// contiguous, so a CTA streams them with TMA: a 128-row tile is 8 regions (64 dims x 128
// rows, 128B-swizzled), region c always lands in slot c of an 8-slot ring, and a slot is
// refilled as soon as the MMAs reading it complete.  Two passes over the tiles:
//  pass 1: S^T = R Q^T per tile (M = 128 rows, N = 64 heads) into TMEM, 64 columns a tile;
//  softmax: the exact per-head maximum over the split, then P^T = 2^(S - max) in bf16, one
//          128-row tile at a time in two buffers, and the per-head sums;
//  pass 2: the same tiles again (L2-resident by then): O^T += R^T P^T (M = 128 dims a chunk,
//          N = 64 heads, K = 128 rows); rows past the split's end (only in its last tile, the
//          one still resident from pass 1 and read first) are zeroed by the softmax warps
//          beside their P^T rows (they may hold anything, and 0 x NaN is NaN).
// Warps 0-7: softmax and epilogue (warp w: TMEM lanes 32 (w & 3) .. +31, heads 32 (w >> 2) ..
// +31; a lane is a row, then a dim); warp 8: TMA producer and TMEM owner; warp 9: MMA issuer.
// The partials (max, sum, unnormalised O) are merged with the sink by attn_merge_wide_kernel.
constexpr int kHdTiles = 4;
constexpr int kHdThreads = 320;
struct HdLayout {
  static constexpr uint32_t kQ = 0;                        // 8 regions x (64 heads x 128 B)
  static constexpr uint32_t kSlot = kRows * 128;           // one region of a tile: 16 KB
  static constexpr uint32_t kRing = kQ + kH * kD * 2;      // 8 slots
  static constexpr uint32_t kP = kRing + 8 * kSlot;        // [2] P^T tiles: 128 rows x 128 B
  static constexpr uint32_t kMisc = kP + 2 * kRows * 128;
  // s_red [4][64], s_max [64], s_sum [64]; 24 barriers; TMEM slot and abort flag
  static constexpr uint32_t kMiscBytes = 6 * kH * 4 + 24 * 8 + 16;
  static constexpr size_t kSmem = 1024 + kMisc + kMiscBytes;
};
static_assert(HdLayout::kSmem <= 232448, "shared memory of one CTA");

struct HdPlan {
  int n_es;      // entry splits of a query (the window split, if any, comes after them)
  int rps;       // entry rows a split: a multiple of 128, at most kHdTiles * 128
  int n_split;   // n_es + (W > 0)
  float* part_o;
  float* part_ml;
};

__global__ void __launch_bounds__(kHdThreads, 1)
    attn_hca_dec_kernel(const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap lmap,
                        const __grid_constant__ CUtensorMap qmap, const AttnArgs a, const HdPlan hp) {
  using LY = HdLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + LY::kQ;
  uint8_t* sRing = smem + LY::kRing;
  uint8_t* sP = smem + LY::kP;
  float* s_red = reinterpret_cast<float*>(smem + LY::kMisc);  // [4][64]
  float* s_max = s_red + 4 * kH;                               // [64]
  float* s_sum = s_max + kH;                                   // [64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_sum + kH);
  uint64_t* full = bars;          // [8] slot landed (producer, tx bytes)
  uint64_t* empty = bars + 8;     // [8] slot read by its MMAs (commit)
  uint64_t* qfull = bars + 16;    // Q landed
  uint64_t* sdone = bars + 17;    // every S^T tile of the split committed
  uint64_t* pfull = bars + 18;    // [2] P^T tile written (256 softmax threads)
  uint64_t* pempty = bars + 20;   // [2] P^T tile read (commit)
  uint64_t* odone = bars + 22;    // every O^T product committed
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + 24);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sTmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int64_t r = blockIdx.y;
  const int b = static_cast<int>(r / a.T);
  const float scale_log2 = a.softmax_scale * kLog2e;

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(qfull, 1);
    mbar_init(sdone, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], 256);
      mbar_init(&pempty[i], 1);
    }
    mbar_init(odone, 1);
    fence_mbar_init();
    *sAbort = 0;
  }
  if (warp == 8) {
    tmem_alloc(sTmem, 512);
    tmem_relinquish();
  }
  // Decode step (a.dense_step): the kernel before this one is the step's compressor, which
  // triggers only after its own wait, so every row but the entry it writes this step is
  // already visible; only the split holding that entry waits, before its last tile.
  if (!a.dense_step) pdl_wait();
  pdl_trigger();
  const int64_t t = a.q_pos[r];
  int n;          // rows of this split
  int64_t row0;   // their first row in the tensor map
  const CUtensorMap* map;
  bool wait_last = false;  // the last tile holds the entry written this step
  if (split < hp.n_es) {
    int64_t nv = t >= 0 ? (t + 1) / a.dense_m : 0;
    nv = nv < a.E_cap ? nv : a.E_cap;
    const int64_t lo = static_cast<int64_t>(split) * hp.rps;
    const int64_t cnt = nv - lo;
    n = cnt <= 0 ? 0 : (cnt < hp.rps ? static_cast<int>(cnt) : hp.rps);
    row0 = static_cast<int64_t>(b) * a.E_cap + lo;
    map = &kvmap;
    wait_last = a.dense_step && n > 0 && (t + 1) % a.dense_m == 0 && (t + 1) / a.dense_m - 1 == lo + n - 1;
  } else {
    const int64_t lbase = a.local_base[b];
    int64_t p_lo;
    window_of(t, a.W, lbase, a.L, p_lo, n);
    row0 = static_cast<int64_t>(b) * a.L + (p_lo - lbase);
    map = &lmap;
  }
  const int nt = (n + kRows - 1) / kRows;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem, tO = tmem + 256;  // S^T of tile i at columns 64 i; O^T chunk cc at 256 + 64 cc

  if (warp == 8) {
    // ---- producer: Q, then the regions of pass 1 and pass 2 in the order the MMAs read them
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(qfull, kH * kD * 2);
      for (int c = 0; c < 8; ++c) tma_load_2d(sQ + c * (kH * 128), &qmap, qfull, 64 * c, static_cast<int>(r * kH));
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      // use u of a slot: pass-1 tile u (u < nt), then pass-2 tile 2 nt - 2 - u (the last
      // tile stays in the ring from pass 1 and is read first in pass 2)
      for (int j = 0; ok && j < 8 * (2 * nt - 1); ++j) {
        const int slot = j & 7, use = j >> 3, tile = use < nt ? use : 2 * nt - 2 - use;
        if (use > 0) ok = mbar_wait(&empty[slot], (use - 1) & 1, a.err, sAbort);
        if (!ok) break;
        if (wait_last && j == 8 * (nt - 1)) pdl_wait();
        mbar_arrive_expect_tx(&full[slot], LY::kSlot);
        const int y = static_cast<int>(row0 + static_cast<int64_t>(tile) * kRows);
        if (use < nt)
          tma_load_2d(sRing + slot * LY::kSlot, map, &full[slot], 64 * slot, y);
        else
          tma_load_2d_hint(sRing + slot * LY::kSlot, map, &full[slot], 64 * slot, y, pol);
      }
    }
  } else if (warp == 9) {
    // ---- MMA issuer (lane 0 issues)
    if (nt > 0) {
      bool ok = __all_sync(0xffffffffu, mbar_wait(qfull, 0, a.err, sAbort));
      const uint32_t ring = smem_u32(sRing), qb = smem_u32(sQ), pb = smem_u32(sP);
      const uint32_t idesc_s = idesc_bf16(kRows, kH, false, false);
      const uint32_t idesc_o = idesc_bf16(kRows, kH, true, true);
      for (int i = 0; ok && i < nt; ++i) {
        for (int c = 0; c < 8; ++c) {
          ok = __all_sync(0xffffffffu, mbar_wait(&full[c], i & 1, a.err, sAbort));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16(tS + 64 * i, smem_desc(ring + c * LY::kSlot + ks * 32, 16, 1024),
                       smem_desc(qb + c * (kH * 128) + ks * 32, 16, 1024), idesc_s, (c | ks) > 0 ? 1u : 0u);
            if (i + 1 < nt) mma_commit(&empty[c]);  // the last tile is read again by pass 2
          }
          __syncwarp();
        }
      }
      if (ok && lane == 0) mma_commit(sdone);
      // pass 2, tiles nt-1 .. 0: the k-th is in P^T buffer k & 1 and (k > 0) in use nt-1+k
      for (int k = 0; ok && k < nt; ++k) {
        const int use = nt - 1 + k;
        ok = __all_sync(0xffffffffu, mbar_wait(&pfull[k & 1], (k >> 1) & 1, a.err, sAbort));
        for (int cc = 0; ok && cc < 4; ++cc) {
          if (k > 0)
            ok = __all_sync(0xffffffffu, mbar_wait(&full[2 * cc], use & 1, a.err, sAbort) &&
                                             mbar_wait(&full[2 * cc + 1], use & 1, a.err, sAbort));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int ks = 0; ks < kRows / 16; ++ks)
              mma_bf16(tO + 64 * cc, smem_desc(ring + (2 * cc) * LY::kSlot + ks * 2048, LY::kSlot, 1024),
                       smem_desc(pb + (k & 1) * (kRows * 128) + ks * 2048, 8192, 1024), idesc_o,
                       (k > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&empty[2 * cc]);
            mma_commit(&empty[2 * cc + 1]);
          }
          __syncwarp();
        }
        if (ok && lane == 0) mma_commit(&pempty[k & 1]);
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(odone);
    }
  } else {
    // ---- softmax and epilogue: warps 0-7, thread = TMEM lane 32 (w & 3) + l, heads hb .. hb+31
    const int qd = warp & 3, hb = 32 * (warp >> 2);
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const int row = qd * 32 + lane;
    float* ml = hp.part_ml + (r * hp.n_split + split) * 2 * kH;
    if (nt > 0) {
      bool ok = named_and(1, 256, mbar_wait(sdone, 0, a.err, sAbort));
      tc_fence_after();
      float mx = -INFINITY;  // of head hb + lane, over the rows this warp's lanes hold
      for (int i = 0; ok && i < nt; ++i) {
        float x[32];
        tmem_ld32(tS + lane_off + 64 * i + hb, x);
        tmem_wait_ld(x);
        const bool valid = i * kRows + row < n;
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = valid ? x[e] * scale_log2 : -INFINITY;
        mx = fmaxf(mx, warp_reduce32<true>(x));
      }
      s_red[qd * kH + hb + lane] = mx;
      named_sync(1, 256);
      if (tid < kH)
        s_max[tid] = fmaxf(fmaxf(s_red[tid], s_red[kH + tid]), fmaxf(s_red[2 * kH + tid], s_red[3 * kH + tid]));
      named_sync(1, 256);
      float mh[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) mh[e] = s_max[hb + e];
      float lsum = 0.f;  // of head hb + lane
      for (int k = 0; ok && k < nt; ++k) {  // tiles in the order pass 2 reads them
        const int i = nt - 1 - k, buf = k & 1;
        if (k >= 2) ok = named_and(1, 256, mbar_wait(&pempty[buf], ((k >> 1) - 1) & 1, a.err, sAbort));
        if (!ok) break;
        float x[32];
        tmem_ld32(tS + lane_off + 64 * i + hb, x);
        tmem_wait_ld(x);
        const bool valid = i * kRows + row < n;
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = valid ? ex2_approx(fmaf(x[e], scale_log2, -mh[e])) : 0.f;
        if (!valid) {  // only in the resident last tile (k = 0): zero the row in the ring, as
                       // pass 2 multiplies it by P = 0 and 0 x NaN is NaN; the S products that
                       // read it completed before the softmax began
#pragma unroll
          for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(sRing + ((hb >> 5) * 4 + g) * LY::kSlot + row * 128 + c * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
        }
        uint8_t* prow = sP + buf * (kRows * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 pk;
          uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 two = __floats2bfloat162_rn(x[c * 8 + 2 * e], x[c * 8 + 2 * e + 1]);
            w[e] = *reinterpret_cast<uint32_t*>(&two);
          }
          *reinterpret_cast<uint4*>(prow + sw128(row, (hb >> 3) + c)) = pk;
        }
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(&pfull[buf]);
        lsum += warp_reduce32<false>(x);
      }
      s_red[qd * kH + hb + lane] = lsum;
      named_sync(1, 256);
      if (tid < kH) {
        ml[tid] = ok ? s_max[tid] : -INFINITY;
        ml[kH + tid] = ok ? (s_red[tid] + s_red[kH + tid]) + (s_red[2 * kH + tid] + s_red[3 * kH + tid]) : 0.f;
      }
      ok = named_and(1, 256, ok && mbar_wait(odone, 0, a.err, sAbort));
      tc_fence_after();
      if (ok) {
        float* po = hp.part_o + (r * hp.n_split + split) * kH * kD;
        for (int cc = 0; cc < 4; ++cc) {
          float v[32];
          tmem_ld32(tO + lane_off + 64 * cc + hb, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int e = 0; e < 32; ++e) po[(hb + e) * kD + cc * 128 + row] = v[e];
        }
      }
    } else if (tid < kH) {
      ml[tid] = -INFINITY;
      ml[kH + tid] = 0.f;
    }
  }
  if (a.dense_step) pdl_wait();  // complete only after the compressor: keeps the stream order
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of many split partials ([query][split][head][dim]) with the sink: one CTA per
// (query, head), thread t owns dims 4t .. 4t+3.  Thread 0 stages the n_split partial rows of
// the head (2 KiB each, contiguous) into shared memory with bulk copies on one mbarrier, all
// in flight at once; meanwhile thread x < n_split reads split x's (m, l) and block reductions
// give M = max(m_x, sink) and den = sum_x l_x 2^(m_x - M) + 2^(sink - M); the staged rows are
// then summed in split order.
constexpr int kMaxSplitDec = 64;  // split partials a query may have
constexpr int kMwThreads = 128;
__global__ void __launch_bounds__(kMwThreads) attn_merge_wide_kernel(const AttnArgs a, const TcAttnSplit sp) {
  extern __shared__ __align__(16) float s_po[];  // [n_split][kD]
  __shared__ float s_f[kMaxSplitDec];
  __shared__ float s_red[kMwThreads / 32];
  __shared__ uint64_t s_bar;
  const int64_t r = blockIdx.x;
  const int h = blockIdx.y;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int ns = sp.n_split;
  if (t == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();
  if (a.sel_seen && h == 0 && t == 0) {  // this step's list consumed
    a.sel_seen[r] = __ldcg(a.sel_done + r);
    if (a.sel_chunks) a.sel_chunks[r] = 0u;
  }
  if (t == 0) {
    mbar_arrive_expect_tx(&s_bar, static_cast<uint32_t>(ns) * kD * 4);
    for (int x = 0; x < ns; ++x) bulk_g2s(s_po + x * kD, sp.part_o + ((r * ns + x) * kH + h) * kD, kD * 4, &s_bar);
  }
  float m = -INFINITY, l = 0.f;
  if (t < ns) {
    m = __ldcg(sp.part_ml + (r * ns + t) * 2 * kH + h);
    l = __ldcg(sp.part_ml + (r * ns + t) * 2 * kH + kH + h);
  }
  const float sk = a.sink[h] * kLog2e;
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_red[warp] = M;
  __syncthreads();  // (also publishes the barrier's initialisation)
  M = sk;
#pragma unroll
  for (int w = 0; w < kMwThreads / 32; ++w) M = fmaxf(M, s_red[w]);
  const float f = m == -INFINITY ? 0.f : exp2f(m - M);
  float part = l * f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  __syncthreads();  // every thread has read s_red
  if (lane == 0) s_red[warp] = part;
  if (t < ns) s_f[t] = f;
  __syncthreads();
  float den = exp2f(sk - M);
#pragma unroll
  for (int w = 0; w < kMwThreads / 32; ++w) den += s_red[w];
  if (t == 0 && a.lse) a.lse[r * kH + h] = (M + log2f(den)) * kLn2;
  mbar_wait(&s_bar, 0, a.err, nullptr);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int x = 0; x < ns; ++x) {
    const float fx = s_f[x];
    if (fx != 0.f) {  // splits without rows wrote no partial
      const float4 v = *reinterpret_cast<const float4*>(s_po + x * kD + 4 * t);
      acc.x = fmaf(v.x, fx, acc.x);
      acc.y = fmaf(v.y, fx, acc.y);
      acc.z = fmaf(v.z, fx, acc.z);
      acc.w = fmaf(v.w, fx, acc.w);
    }
  }
  const float inv = 1.f / den;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + (r * kH + h) * kD + 4 * t) = pk;
}

// The merge of sp.n_split (<= kMaxSplitDec) partials a query.
cudaError_t launch_merge_wide(const AttnArgs& a, const TcAttnSplit& sp, int64_t rows, cudaStream_t s) {
  static std::atomic<unsigned long long> mattr{0};
  if (first_use_in_context(mattr))
    cudaFuncSetAttribute(attn_merge_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSplitDec * kD * 4);
  const cudaError_t e = launch_pdl(attn_merge_wide_kernel, dim3(static_cast<unsigned>(rows), kH), dim3(kMwThreads),
                                   static_cast<size_t>(sp.n_split) * kD * 4, s, a, sp);
  count_launches(1);
  return e;
}

bool attn_uses_tensor_cores(int act, int H, int d, int k) {
  return act == CSA_BF16 && H == kH && d == kD && k <= kMaxK;
}

TcAttnSplit plan_split(int B, int T, int k, int W, int num_sms) {
  TcAttnSplit s{};
  const int64_t rows = static_cast<int64_t>(B) * T;
  const int max_rows = k + W;
  if (rows < num_sms && max_rows > kRows) {
    s.rows_per_split = kRows;
    s.n_split = (max_rows + kRows - 1) / kRows;
    if (s.n_split > kMaxSplit) {
      s.rows_per_split = ((max_rows + kMaxSplit - 1) / kMaxSplit + kRows - 1) / kRows * kRows;
      s.n_split = (max_rows + s.rows_per_split - 1) / s.rows_per_split;
    }
  } else {
    s.rows_per_split = max_rows;
    s.n_split = 1;
  }
  return s;
}

// Dense rows (HCA): few queries split their rows over CTAs of attn_pf_kernel so that the
// grid fills the SMs once (rows_per_split a multiple of the 64-row tile, at most
// kMaxSplitDec splits); many queries take one CTA each.
TcAttnSplit plan_dense(int64_t rows, int64_t max_rows, int num_sms) {
  TcAttnSplit s{};
  s.n_split = 1;
  s.rows_per_split = 0;
  if (rows >= num_sms || max_rows <= 2 * kPR) return s;
  const int64_t want = num_sms / rows;  // >= 1
  int64_t rps = (max_rows + want - 1) / want;
  const int64_t lo = (max_rows + kMaxSplitDec - 1) / kMaxSplitDec;
  if (rps < lo) rps = lo;
  if (rps < 2 * kPR) rps = 2 * kPR;
  rps = (rps + kPR - 1) / kPR * kPR;
  const int64_t ns = (max_rows + rps - 1) / rps;
  if (ns > 1) {
    s.n_split = static_cast<int>(ns);
    s.rows_per_split = static_cast<int>(rps);
  }
  return s;
}

bool dense_uses_tensor_cores(int act, int H, int d) { return act == CSA_BF16 && H == kH && d == kD; }

// attn_hca_dec_kernel's plan for few queries: about num_sms / rows CTAs a query (one of them
// for the window), entry splits of a multiple of 128 rows, at most kHdTiles tiles and
// kMaxSplitDec splits; n_split = 0 when the entries do not fit that.  (Splits of any multiple
// of 16 rows that fill every SM measured slower: their partial last tiles cost more in pass 2
// than the extra CTAs gain.)
HdPlan plan_hca_dec(int64_t rows, int64_t E_cap, int W, int num_sms) {
  HdPlan p{};
  if (rows >= num_sms) return p;
  const int win = W > 0 ? 1 : 0;
  const int64_t want = std::max<int64_t>(1, num_sms / rows - win);
  int64_t rps = (E_cap + want - 1) / want;
  rps = std::max<int64_t>(rps, (E_cap + (kMaxSplitDec - win) - 1) / (kMaxSplitDec - win));
  rps = std::max<int64_t>((rps + kRows - 1) / kRows * kRows, kRows);
  if (rps > kHdTiles * kRows) return p;
  p.rps = static_cast<int>(rps);
  p.n_es = static_cast<int>((E_cap + rps - 1) / rps);
  p.n_split = p.n_es + win;
  return p;
}

size_t dense_partials_bytes(int64_t rows, int n_split) {
  return align_up(static_cast<size_t>(rows * n_split * kH * kD) * 4, 256) +
         align_up(static_cast<size_t>(rows * n_split * 2 * kH) * 4, 256);
}

}  // namespace

size_t attn_dense_workspace_bytes(int B, int T, int H, int d, int64_t E_cap, int W, int act, int num_sms) {
  if (!dense_uses_tensor_cores(act, H, d)) return 0;
  const int64_t rows = static_cast<int64_t>(B) * T;
  const HdPlan hp = plan_hca_dec(rows, E_cap, W, num_sms);
  if (hp.n_split > 0) return dense_partials_bytes(rows, hp.n_split);
  const TcAttnSplit s = plan_dense(rows, E_cap + W, num_sms);
  if (s.n_split == 1) return 0;
  return dense_partials_bytes(rows, s.n_split);
}

// The decode split plan with at least min_split splits (candidate mode of the decode step).
TcAttnSplit plan_split_min(int B, int T, int k, int W, int num_sms, int min_split) {
  TcAttnSplit s = plan_split(B, T, k, W, num_sms);
  if (s.n_split > 1 && s.rows_per_split == kRows && min_split > s.n_split) s.n_split = min_split;
  return s;
}

size_t attn_workspace_bytes(int B, int T, int H, int d, int k, int W, int act, int num_sms, int min_split) {
  if (!attn_uses_tensor_cores(act, H, d, k)) return 0;
  const TcAttnSplit s = plan_split_min(B, T, k, W, num_sms, min_split);
  if (s.n_split == 1) return 0;
  const int64_t rows = static_cast<int64_t>(B) * T;
  return align_up(static_cast<size_t>(rows * s.n_split * kH * kD) * 4, 256) +
         align_up(static_cast<size_t>(rows * s.n_split * 2 * kH) * 4, 256);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T;
  if (rows == 0) return cudaSuccess;
  if (a.dense_m > 0 && dense_uses_tensor_cores(a.act, a.H, a.d)) {
    HdPlan hp = plan_hca_dec(rows, a.E_cap, a.W, a.num_sms);
    if (hp.n_split > 0) {
      uint8_t* ws = static_cast<uint8_t*>(a.ws);
      hp.part_o = reinterpret_cast<float*>(ws);
      hp.part_ml = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(rows * hp.n_split * kH * kD) * 4, 256));
      CUtensorMap kvmap, lmap, qmap;
      const uint64_t kv_rows = std::max<int64_t>(1, static_cast<int64_t>(a.B) * a.E_cap);
      const uint64_t l_rows = std::max<int64_t>(1, static_cast<int64_t>(a.B) * a.L);
      if (!encode_tmap_2d(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(a.kv_comp), kD, kv_rows,
                          kD * 2, 64, kRows) ||
          !encode_tmap_2d(&lmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(a.kv_local), kD, l_rows, kD * 2,
                          64, kRows) ||
          !encode_tmap_2d(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void*>(a.q), kD,
                          static_cast<uint64_t>(rows) * kH, kD * 2, 64, kH))
        return cudaErrorInvalidValue;
      static std::atomic<unsigned long long> hattr{0};
      if (first_use_in_context(hattr)) {
        cudaFuncSetAttribute(attn_hca_dec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(HdLayout::kSmem));
      }
      cudaError_t e = launch_pdl(attn_hca_dec_kernel, dim3(hp.n_split, static_cast<unsigned>(rows)),
                                 dim3(kHdThreads), HdLayout::kSmem, s, kvmap, lmap, qmap, a, hp);
      count_launches(1);
      if (e != cudaSuccess) return e;
      TcAttnSplit sp{};
      sp.n_split = hp.n_split;
      sp.rows_per_split = hp.rps;
      sp.part_o = hp.part_o;
      sp.part_ml = hp.part_ml;
      return launch_merge_wide(a, sp, rows, s);
    }
    TcAttnSplit sp = plan_dense(rows, a.E_cap + a.W, a.num_sms);
    if (sp.n_split > 1) {
      uint8_t* ws = static_cast<uint8_t*>(a.ws);
      sp.part_o = reinterpret_cast<float*>(ws);
      sp.part_ml = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(rows * sp.n_split * kH * kD) * 4, 256));
    }
    static std::atomic<unsigned long long> dattr{0};
    if (first_use_in_context(dattr)) {
      cudaFuncSetAttribute(attn_pf_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(PfLayout::kSmem));
    }
    cudaError_t e = launch_pdl(attn_pf_kernel<0>, dim3(static_cast<unsigned>(rows), sp.n_split), dim3(kPfThreads),
                               PfLayout::kSmem, s, a, sp);
    count_launches(1);
    if (e != cudaSuccess || sp.n_split == 1) return e;
    return launch_merge_wide(a, sp, rows, s);
  }
  if (attn_uses_tensor_cores(a.act, a.H, a.d, a.k)) {
    TcAttnSplit sp = plan_split_min(a.B, a.T, a.k, a.W, a.num_sms, a.min_split);
    if (sp.n_split > 1) {
      uint8_t* ws = static_cast<uint8_t*>(a.ws);
      sp.part_o = reinterpret_cast<float*>(ws);
      sp.part_ml = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(rows * sp.n_split * kH * kD) * 4, 256));
    }
    const size_t smem = 1024 + kMiscOff + (kH * 7 + 32) * 4 + 64 + static_cast<size_t>(kMaxK) * 4;
    static std::atomic<unsigned long long> attr{0};
    if (first_use_in_context(attr)) {
      cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    }
    if (sp.n_split == 1 && a.k <= kPfMaxK) {
      static std::atomic<unsigned long long> pattr{0};
      if (first_use_in_context(pattr)) {
        cudaFuncSetAttribute(attn_pf_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(PfLayout::kSmem));
      }
      const cudaError_t e = launch_pdl(attn_pf_kernel<0>, dim3(static_cast<unsigned>(rows)), dim3(kPfThreads),
                                       PfLayout::kSmem, s, a, sp);
      count_launches(1);
      return e;
    }
    if (sp.n_split == 1 || sp.rows_per_split != kRows) {
      const cudaError_t e = launch_pdl(attn_tc_kernel, dim3(sp.n_split, static_cast<unsigned>(rows)),
                                       dim3(kTcThreads), smem, s, a, sp);
      count_launches(1);
      if (e != cudaSuccess || sp.n_split == 1) return e;
      const cudaError_t e2 = launch_pdl(attn_merge_kernel, dim3(static_cast<unsigned>(rows), kH / kMergeHeads),
                                        dim3(kD), 0, s, a, sp);
      count_launches(1);
      return e2;
    }
    // decode: head groups so that split x group x query fills the SMs once
    const int64_t per = static_cast<int64_t>(sp.n_split) * rows;
    const int hg = per * 4 <= a.num_sms ? 4 : (per * 2 <= a.num_sms ? 2 : 1);
    static std::atomic<unsigned long long> dattr{0};
    if (first_use_in_context(dattr)) {
      cudaFuncSetAttribute(attn_dec_kernel<16, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(DecLayout<16>::kSmem));
      cudaFuncSetAttribute(attn_dec_kernel<32, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(DecLayout<32>::kSmem));
      cudaFuncSetAttribute(attn_dec_kernel<64, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(DecLayout<64>::kSmem));
    }
    dim3 grid(sp.n_split, hg, static_cast<unsigned>(rows));
    cudaError_t e =
        hg == 4 ? launch_pdl(attn_dec_kernel<16, 0>, grid, dim3(kTcThreads), DecLayout<16>::kSmem, s, a, sp)
        : hg == 2 ? launch_pdl(attn_dec_kernel<32, 0>, grid, dim3(kTcThreads), DecLayout<32>::kSmem, s, a, sp)
                  : launch_pdl(attn_dec_kernel<64, 0>, grid, dim3(kTcThreads), DecLayout<64>::kSmem, s, a, sp);
    count_launches(1);
    if (e != cudaSuccess) return e;
    return launch_merge_wide(a, sp, rows, s);
  }
  const size_t smem = (static_cast<size_t>(a.H) * a.d * 2 + kSimtTile * (a.d + 1) + a.H * kSimtTile + 3 * a.H + 32) * 4 +
                      static_cast<size_t>(a.k) * 4;
  cudaError_t e;
  if (a.act == CSA_F32) {
    cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    e = launch_pdl(attn_simt_kernel<float>, dim3(static_cast<unsigned>(rows)), dim3(kSimtThreads), smem, s, a);
  } else {
    cudaFuncSetAttribute(attn_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    e = launch_pdl(attn_simt_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(rows)), dim3(kSimtThreads), smem, s, a);
  }
  count_launches(1);
  return e;
}

bool attn_fp8kv_supported(int B, int T, int H, int d, int k, int W, int act, int num_sms) {
  if (!attn_uses_tensor_cores(act, H, d, k)) return false;
  const TcAttnSplit sp = plan_split(B, T, k, W, num_sms);
  return sp.n_split > 1 && sp.rows_per_split == kRows;
}

// Quantised entries: the decode split plan (few queries), or one CTA a query over its whole
// row list (many queries: the prefill chunk) on attn_pf_kernel.
static bool attn_quantkv_pf(int B, int T, int H, int d, int k, int W, int act, int num_sms) {
  if (!attn_uses_tensor_cores(act, H, d, k)) return false;
  return plan_split(B, T, k, W, num_sms).n_split == 1 && k <= kPfMaxK;
}

bool attn_quantkv_supported(int B, int T, int H, int d, int k, int W, int act, int num_sms) {
  return attn_fp8kv_supported(B, T, H, d, k, W, act, num_sms) || attn_quantkv_pf(B, T, H, d, k, W, act, num_sms);
}

template <int KVF>
cudaError_t launch_attn_quantkv(const AttnArgs& a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T;
  if (rows == 0) return cudaSuccess;
  if (!attn_fp8kv_supported(a.B, a.T, a.H, a.d, a.k, a.W, a.act, a.num_sms)) {
    if (!attn_quantkv_pf(a.B, a.T, a.H, a.d, a.k, a.W, a.act, a.num_sms)) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> pattr{0};
    if (first_use_in_context(pattr))
      cudaFuncSetAttribute(attn_pf_kernel<KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(PfLayout::kSmem));
    const TcAttnSplit sp1 = plan_split(a.B, a.T, a.k, a.W, a.num_sms);
    const cudaError_t e = launch_pdl(attn_pf_kernel<KVF>, dim3(static_cast<unsigned>(rows)), dim3(kPfThreads),
                                     PfLayout::kSmem, s, a, sp1);
    count_launches(1);
    return e;
  }
  TcAttnSplit sp = plan_split_min(a.B, a.T, a.k, a.W, a.num_sms, a.min_split);
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  sp.part_o = reinterpret_cast<float*>(ws);
  sp.part_ml = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(rows * sp.n_split * kH * kD) * 4, 256));
  const int64_t per = static_cast<int64_t>(sp.n_split) * rows;
  const int hg = per * 4 <= a.num_sms ? 4 : (per * 2 <= a.num_sms ? 2 : 1);
  static std::atomic<unsigned long long> fattr{0};
  if (first_use_in_context(fattr)) {
    cudaFuncSetAttribute(attn_dec_kernel<16, KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(DecLayout<16>::kSmem));
    cudaFuncSetAttribute(attn_dec_kernel<32, KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(DecLayout<32>::kSmem));
    cudaFuncSetAttribute(attn_dec_kernel<64, KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(DecLayout<64>::kSmem));
  }
  dim3 grid(sp.n_split, hg, static_cast<unsigned>(rows));
  cudaError_t e =
      hg == 4 ? launch_pdl(attn_dec_kernel<16, KVF>, grid, dim3(kTcThreads), DecLayout<16>::kSmem, s, a, sp)
      : hg == 2 ? launch_pdl(attn_dec_kernel<32, KVF>, grid, dim3(kTcThreads), DecLayout<32>::kSmem, s, a, sp)
                : launch_pdl(attn_dec_kernel<64, KVF>, grid, dim3(kTcThreads), DecLayout<64>::kSmem, s, a, sp);
  count_launches(1);
  if (e != cudaSuccess) return e;
  return launch_merge_wide(a, sp, rows, s);
}

cudaError_t launch_attn_fp8kv(const AttnArgs& a, cudaStream_t s) { return launch_attn_quantkv<1>(a, s); }
cudaError_t launch_attn_mxfp4kv(const AttnArgs& a, cudaStream_t s) { return launch_attn_quantkv<2>(a, s); }

}  // namespace csa
