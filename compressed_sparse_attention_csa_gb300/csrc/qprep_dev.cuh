// Query operand of the tensor-core indexer, one (query, head) row per warp.
//
// Each query group's image is the exact shared-memory layout the indexer kernel pulls with
// one bulk copy: [b_bytes: B operand, 128B-swizzled K-major][w_bytes: the gates].  bf16 keys:
// the bf16 query row as two 64-element regions.  E4M3 keys: the row scaled by s = amax/448 and
// split into two E4M3 terms hi + lo (hi = e4m3(q/s), lo = e4m3(q/s - hi)), and the gate stored
// as w * s, since s > 0 factors out of the ReLU.
//
// Used by the standalone query-prep kernel and by the decode step's compressor launch.
#pragma once
#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {

template <bool FP8>
__device__ __forceinline__ void qprep_row(const IndexerArgs& a, const IndexerLayout& L, uint8_t* images, int qg,
                                          int b, int gh, int lane) {
  const int HI = a.HI, G = L.G, N = L.N, T = a.T;
  const int g0 = qg * G;
  const int64_t qrow0 = static_cast<int64_t>(b) * T + g0;
  uint8_t* img = images + (static_cast<size_t>(b) * L.n_qgroups + qg) * (L.b_bytes + L.w_bytes);
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

}  // namespace csa
