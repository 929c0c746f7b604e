// Query operand of the tensor-core indexer, one (query, head) row per warp.
//
// Each query group's image is the exact shared-memory layout the indexer kernel pulls with
// one bulk copy: [b_bytes: B operand, 128B-swizzled K-major][w_bytes: the gates].  bf16 keys:
// the bf16 query row as two 64-element regions.  E4M3 keys: the row scaled by s = amax/448 and
// split into two E4M3 terms hi + lo (hi = e4m3(q/s), lo = e4m3(q/s - hi)), and the gate stored
// as w * s, since s > 0 factors out of the ReLU.
//
// Used by the standalone query-prep kernel, the compressor launch, and the decode-step
// indexer (which writes the image straight into its shared memory).
#pragma once
#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {

// img: this query group's image (global workspace, or the indexer CTA's shared memory).
template <bool FP8>
__device__ __forceinline__ void qprep_row(const IndexerArgs& a, const IndexerLayout& L, uint8_t* img, int qg,
                                          int b, int gh, int lane) {
  const int HI = a.HI, G = L.G, N = L.N, T = a.T;
  const int g0 = qg * G;
  const int64_t qrow0 = static_cast<int64_t>(b) * T + g0;
  float* wimg = reinterpret_cast<float*>(img + L.b_bytes);
  const __nv_bfloat16* qI = static_cast<const __nv_bfloat16*>(a.qI);
  const int g = gh / HI, h = gh - g * HI;
  const bool valid = g0 + g < T;
  if constexpr (!FP8) {
    // 256-byte bf16 row: even lane l copies 16-byte chunk l/2, as two regions of 64 elements
    const int c = lane >> 1;  // 0..15
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (valid && (lane & 1) == 0) v = *reinterpret_cast<const uint4*>(qI + ((qrow0 + g) * HI + h) * 128 + c * 8);
    if ((lane & 1) == 0) *reinterpret_cast<uint4*>(img + (c >> 3) * (N * 128) + sw128(gh, c & 7)) = v;
    if (lane == 0) wimg[gh] = valid ? a.w[(qrow0 + g) * HI + h] : 0.f;
  } else {
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    float wv = 0.f;
    if (valid) {
      const uint2 raw = *reinterpret_cast<const uint2*>(qI + ((qrow0 + g) * HI + h) * 128 + lane * 4);
      if (lane == 0) wv = a.w[(qrow0 + g) * HI + h];
      const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      x[0] = __low2float(p0);
      x[1] = __high2float(p0);
      x[2] = __low2float(p1);
      x[3] = __high2float(p1);
    }
    float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float sc = am > 0.f ? am / 448.f : 1.f;
    const float inv = 1.f / sc;
    uint32_t hi4 = 0u, lo4 = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float y = x[j] * inv;
      const uint8_t ch = f_to_e4m3(y);
      const uint8_t cl = f_to_e4m3(y - e4m3_to_f(ch));
      hi4 |= static_cast<uint32_t>(ch) << (8 * j);
      lo4 |= static_cast<uint32_t>(cl) << (8 * j);
    }
    const uint32_t off = sw128(gh, lane >> 2) + (lane & 3) * 4;
    *reinterpret_cast<uint32_t*>(img + off) = hi4;
    *reinterpret_cast<uint32_t*>(img + N * 128 + off) = lo4;
    if (lane == 0) wimg[gh] = wv * sc;
  }
}

__device__ __forceinline__ uint8_t* qprep_image(const IndexerLayout& L, uint8_t* images, int qg, int b) {
  return images + (static_cast<size_t>(b) * L.n_qgroups + qg) * (L.b_bytes + L.w_bytes);
}

// ---- decode step, inside the indexer launch -----------------------------------------

// NC channels of the compressed entry the token t completes ("DeepSeek V4-Flash: The Cost of
// Deciding What to Read", section "The compressor has two streams and they overlap"): the
// tail holds tokens t-2m+1..t, so stream a (current block) is rows m..2m-1 and stream b
// (previous block) rows 0..m-1; a softmax over the 2m gate logits plus the positional bias,
// then the weighted sum of the values.  has_b = false (entry 0) keeps stream a only.  MT
// bounds 2m at compile time so every load of every channel is in flight at once.
template <typename T, int MT, int NC>
__device__ __forceinline__ void compress_tail(const T* kv, const T* z, const float* bias, int m, int dim,
                                              const int (&c)[NC], bool has_b, float (&out)[NC]) {
  // every load first (tokens past the block read its first row and are dropped below), so
  // that they are in flight together; the bias is added once they have landed
  float lg[NC][MT], val[NC][MT], bs[NC][MT];
#pragma unroll
  for (int j = 0; j < MT; ++j) {
    const bool in = j < 2 * m && (j < m || has_b);
    const int st = in && j >= m ? 1 : 0;
    const int jj = !in ? 0 : (j < m ? j : j - m);
    const int64_t row = static_cast<int64_t>((st == 0 ? m : 0) + jj) * 2 + st;
#pragma unroll
    for (int n = 0; n < NC; ++n) {
      lg[n][j] = load_f<T>(z + row * dim + c[n]);
      bs[n][j] = bias[(st * m + jj) * dim + c[n]];
      val[n][j] = load_f<T>(kv + row * dim + c[n]);
    }
  }
#pragma unroll
  for (int j = 0; j < MT; ++j)
#pragma unroll
    for (int n = 0; n < NC; ++n) lg[n][j] += bs[n][j];
  const int nt = has_b ? 2 * m : m;
#pragma unroll
  for (int n = 0; n < NC; ++n) {
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < MT; ++j)
      if (j < nt) mx = fmaxf(mx, lg[n][j]);
    float sum = 0.f, acc = 0.f;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      if (j < nt) {
        const float e = expf(lg[n][j] - mx);
        sum += e;
        acc = fmaf(e, val[n][j], acc);
      }
    }
    out[n] = acc / sum;
  }
}

// m <= 8 (the fused decode path's limit): 2m <= 16 tokens.
template <int NC>
__device__ __forceinline__ void compress_tail_any(const void* kv, const void* z, const float* bias, bool bf16, int m,
                                                  int dim, const int (&c)[NC], bool has_b, float (&out)[NC]) {
#define CSA_TAIL(T, MT) \
  compress_tail<T, MT, NC>(static_cast<const T*>(kv), static_cast<const T*>(z), bias, m, dim, c, has_b, out)
  if (bf16) {
    if (m <= 4) CSA_TAIL(__nv_bfloat16, 8); else CSA_TAIL(__nv_bfloat16, 16);
  } else {
    if (m <= 4) CSA_TAIL(float, 8); else CSA_TAIL(float, 16);
  }
#undef CSA_TAIL
}

// The new indexer-key entry e of sequence b (dI = 128), by 128 threads (one channel each,
// t128 = 0..127, named barrier `bar`), stored as the compressor stores it: KF = 1, e4m3 codes
// with one fp32 scale (amax/448); KF = 2, MXFP4 (per warp = block of 32 channels one UE8M0
// scale byte, E2M1 codes two to a byte); KF = 0, bf16.  Returns the fp32 scale (1 unless
// e4m3).  Every thread fences its global writes for the TMA loads of the same row that follow
// in this CTA.
template <int KF>
__device__ __forceinline__ float decode_new_key(const IndexerArgs& a, int b, int64_t e, int t128, float* red4,
                                                int bar) {
  const DecodeFuse& f = a.fuse;
  const int dI = a.dI, m = a.m;
  const size_t elem = f.act_bf16 ? 2 : 4;
  const size_t tail = static_cast<size_t>(b) * 2 * m * 2 * dI * elem;
  const int c[1] = {t128};
  float v[1];
  compress_tail_any<1>(static_cast<const uint8_t*>(f.kvI_tail) + tail, static_cast<const uint8_t*>(f.zI_tail) + tail,
                       f.biasI, f.act_bf16, m, dI, c, e > 0, v);
  const int64_t row = static_cast<int64_t>(b) * a.E_cap + e;
  float scale = 1.f;
  if constexpr (KF == 2) {
    float am = fabsf(v[0]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const uint32_t sb = mx_e2m1_scale_byte(am);
    const uint32_t code = e2m1_code(__fdiv_rn(v[0], ue8m0_value(sb)));
    const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
    if ((t128 & 1) == 0)
      static_cast<uint8_t*>(const_cast<void*>(a.kI))[row * (dI / 2) + t128 / 2] = static_cast<uint8_t>(code | (hi << 4));
    if ((t128 & 31) == 0)
      static_cast<uint8_t*>(const_cast<void*>(a.kscale))[row * (dI / 32) + t128 / 32] = static_cast<uint8_t>(sb);
  } else if constexpr (KF == 1) {
    float am = fabsf(v[0]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if ((t128 & 31) == 0) red4[t128 >> 5] = am;
    asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
    am = fmaxf(fmaxf(red4[0], red4[1]), fmaxf(red4[2], red4[3]));
    scale = am > 0.f ? __fdiv_rn(am, 448.f) : 1.f;
    static_cast<uint8_t*>(const_cast<void*>(a.kI))[row * dI + t128] = f_to_e4m3(__fdiv_rn(v[0], scale));
    if (t128 == 0) static_cast<float*>(const_cast<void*>(a.kscale))[row] = scale;
  } else {
    static_cast<__nv_bfloat16*>(const_cast<void*>(a.kI))[row * dI + t128] = __float2bfloat16_rn(v[0]);
  }
  fence_proxy_async_global();
  asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
  return scale;
}

// The new main-KV entry e of sequence b (d <= 512, d % 16 == 0), its channels split over the
// n_parts CTAs that score the sequence's keys in contiguous ranges of `chunk` channels (a
// multiple of 16: whole sectors of the tails, and an MXFP4 block of 16 channels stays inside
// one CTA and one half-warp), one channel a thread (t256 = 0..255), so no CTA holds its key
// stream back for the whole entry.  Stored in the cache's format: the activation dtype; FP8
// entries (e4m3 codes of dims < d - 64, then the last 64 in bf16); or MXFP4 entries (per 16
// channels scale = e4m3(amax / 6), codes = nearest E2M1 of x / scale, two to a byte; the d/2
// payload bytes, then the d/16 scale bytes).
__device__ __forceinline__ void decode_new_kv(const IndexerArgs& a, int b, int64_t e, int t256, int part,
                                              int n_parts) {
  const DecodeFuse& f = a.fuse;
  const int d = f.d, m = a.m;
  const int chunk = ((d + n_parts - 1) / n_parts + 15) & ~15;
  const int c_lo = part * chunk, c_hi = min(d, c_lo + chunk);
  if (c_lo >= d) return;  // uniform across the CTA
  const size_t elem = f.act_bf16 ? 2 : 4;
  const size_t tail = static_cast<size_t>(b) * 2 * m * 2 * d * elem;
  const int64_t row = static_cast<int64_t>(b) * a.E_cap + e;
  for (int c0 = c_lo; c0 < c_hi; c0 += 256) {  // uniform loop: every lane reaches the shuffles
    const int ch = c0 + t256;
    const bool live = ch < c_hi;
    float v = 0.f;
    if (live) {
      const int c[1] = {ch};
      float o[1];
      compress_tail_any<1>(static_cast<const uint8_t*>(f.kv_tail) + tail,
                           static_cast<const uint8_t*>(f.z_tail) + tail, f.bias, f.act_bf16, m, d, c, e > 0, o);
      v = o[0];
    }
    if (f.kv_fmt == 2) {
      // one MXFP4 block = 16 consecutive channels = the 16 lanes of a half-warp
      float am = fabsf(v);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
      const uint8_t sc_code = f_to_e4m3(__fdiv_rn(am, 6.f));
      const float sc = e4m3_to_f(sc_code);
      const uint32_t code = sc > 0.f ? e2m1_code(__fdiv_rn(v, sc)) : 0u;
      const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
      uint8_t* row4 = static_cast<uint8_t*>(f.kv_comp) + row * (d / 2 + d / 16);
      if (live && (ch & 1) == 0) row4[ch / 2] = static_cast<uint8_t>(code | (hi << 4));
      if (live && (ch & 15) == 0) row4[d / 2 + ch / 16] = sc_code;
    } else if (live && f.kv_fmt == 1) {
      uint8_t* row8 = static_cast<uint8_t*>(f.kv_comp) + row * (d + 64);
      if (ch < d - 64)
        row8[ch] = f_to_e4m3(v);
      else
        reinterpret_cast<__nv_bfloat16*>(row8 + d - 64)[ch - (d - 64)] = __float2bfloat16_rn(v);
    } else if (live) {
      if (f.act_bf16)
        static_cast<__nv_bfloat16*>(f.kv_comp)[row * d + ch] = __float2bfloat16_rn(v);
      else
        static_cast<float*>(f.kv_comp)[row * d + ch] = v;
    }
  }
}

// The query image of sequence b (one query, N = HI <= 128 rows) written by 256 threads
// straight into shared memory: 4 threads per head row, 32 dims each; the same arithmetic
// as qprep_row.  img = B operand, followed by the gates.
template <bool FP8>
__device__ __forceinline__ void build_image_cta(const IndexerArgs& a, const IndexerLayout& L, uint8_t* img, int b,
                                                int t256) {
  const int N = L.N;
  const __nv_bfloat16* qI = static_cast<const __nv_bfloat16*>(a.qI) + static_cast<int64_t>(b) * a.HI * 128;
  const float* w = a.w + static_cast<int64_t>(b) * a.HI;
  float* wimg = reinterpret_cast<float*>(img + L.b_bytes);
  constexpr int kRowsPer = 2;  // N <= 128 = 2 x 64
  uint4 raw[kRowsPer][4];
  float wv[kRowsPer];
  const int part = t256 & 3;  // dims 32*part .. 32*part + 31
#pragma unroll
  for (int rr = 0; rr < kRowsPer; ++rr) {
    const int gh = (t256 >> 2) + 64 * rr;
    if (gh < N) {
#pragma unroll
      for (int q = 0; q < 4; ++q) raw[rr][q] = *reinterpret_cast<const uint4*>(qI + gh * 128 + part * 32 + q * 8);
      wv[rr] = w[gh];
    }
  }
#pragma unroll
  for (int rr = 0; rr < kRowsPer; ++rr) {
    const int gh = (t256 >> 2) + 64 * rr;
    if (gh >= N) continue;  // uniform across the 4 threads of a row
    if constexpr (!FP8) {
      // dims 32*part.. = region (part >> 1), 16-byte chunks 4*(part & 1) .. +3
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(img + (part >> 1) * (N * 128) + sw128(gh, 4 * (part & 1) + q)) = raw[rr][q];
      if (part == 0) wimg[gh] = wv[rr];
    } else {
      float x[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[rr][q]);
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          x[q * 8 + 2 * e2] = __low2float(p2[e2]);
          x[q * 8 + 2 * e2 + 1] = __high2float(p2[e2]);
        }
      }
      float am = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) am = fmaxf(am, fabsf(x[j]));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      const float sc = am > 0.f ? am / 448.f : 1.f;
      const float inv = 1.f / sc;
      // 32 codes = two 16-byte chunks (2*part, 2*part + 1) of the 128-byte row, hi then lo
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t hi4[4], lo4[4];
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          hi4[wd] = 0u;
          lo4[wd] = 0u;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float y = x[ch * 16 + wd * 4 + j] * inv;
            const uint8_t chh = f_to_e4m3(y);
            const uint8_t cl = f_to_e4m3(y - e4m3_to_f(chh));
            hi4[wd] |= static_cast<uint32_t>(chh) << (8 * j);
            lo4[wd] |= static_cast<uint32_t>(cl) << (8 * j);
          }
        }
        const uint32_t off = sw128(gh, 2 * part + ch);
        *reinterpret_cast<uint4*>(img + off) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
        *reinterpret_cast<uint4*>(img + N * 128 + off) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
      }
      if (part == 0) wimg[gh] = wv[rr] * sc;
    }
  }
}

}  // namespace csa
