// Gated two-stream KV compression.
//
// "DeepSeek V4-Flash: The Cost of Deciding What to Read", section "The compressor has two
// streams and they overlap": compressed entry i draws stream a (C^a, gate Z^a) from tokens
// [m*i, m*(i+1)) and stream b (C^b, Z^b) from [m*(i-1), m*i); a softmax over those 2m
// gate logits, with the learnable positional bias B^a / B^b added by position inside the
// block, runs independently for every channel, and the entry is the weighted sum of the
// matching C values.  Entry 0 has no previous block and mixes the m stream-a tokens only.
//
// Bandwidth-bound: one CTA per (entry, sequence), one thread per channel group; the softmax
// is taken online in one pass over the 2m tokens in fp32.  An E4M3 output gets one fp32 scale
// per entry (amax/448, codes rounded to nearest, saturating).
#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxPerThread = 8;  // dim <= 1024

template <typename T>
__global__ void __launch_bounds__(kThreads) compress_kernel(CompressArgs a) {
  const int b = blockIdx.y;
  int64_t entry, tok0;
  const int m = a.m;
  if (a.q_pos) {
    const int64_t t = a.q_pos[b];
    if ((t + 1) % m != 0) return;
    entry = (t + 1) / m - 1;
    tok0 = t - 2 * m + 1;
  } else {
    entry = a.ent_begin + blockIdx.x;
    tok0 = a.tok0;
  }
  if (entry < 0 || entry >= a.E_cap) return;
  const int64_t n_tok = a.q_pos ? 2 * m : a.n_tok;
  const int dim = a.dim;
  const T* kv = static_cast<const T*>(a.kv) + static_cast<int64_t>(b) * n_tok * 2 * dim;
  const T* z = static_cast<const T*>(a.z) + static_cast<int64_t>(b) * n_tok * 2 * dim;

  float vals[kMaxPerThread];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < kMaxPerThread; ++u) {
    const int c = threadIdx.x + u * kThreads;
    vals[u] = 0.f;
    if (c >= dim) continue;
    float mx = -INFINITY, sum = 0.f, acc = 0.f;
    // stream a: the current block; stream b: the previous block (absent for entry 0)
    for (int st = 0; st < 2; ++st) {
      if (st == 1 && entry == 0) break;
      const int64_t first_tok = (st == 0) ? m * entry : m * (entry - 1);
      for (int j = 0; j < m; ++j) {
        const int64_t r = first_tok + j - tok0;
        const int64_t off = (r * 2 + st) * dim + c;
        const float lg = load_f<T>(z + off) + a.bias[(st * m + j) * dim + c];
        const float v = load_f<T>(kv + off);
        if (lg > mx) {
          const float sc = expf(mx - lg);  // 0 on the first token
          sum = sum * sc + 1.f;
          acc = acc * sc + v;
          mx = lg;
        } else {
          const float e = expf(lg - mx);
          sum += e;
          acc = fmaf(e, v, acc);
        }
      }
    }
    vals[u] = acc / sum;
    amax = fmaxf(amax, fabsf(vals[u]));
  }

  const int64_t row = static_cast<int64_t>(b) * a.E_cap + entry;
  if (a.out_dtype == CSA_E4M3) {
    __shared__ float s_red[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    float am = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) am = fmaxf(am, s_red[w]);
    const float scale = am > 0.f ? __fdiv_rn(am, 448.f) : 1.f;
    uint8_t* o = static_cast<uint8_t*>(a.out) + row * dim;
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = threadIdx.x + u * kThreads;
      if (c < dim) o[c] = f_to_e4m3(__fdiv_rn(vals[u], scale));
    }
    if (threadIdx.x == 0) a.out_scale[row] = scale;
  } else if (a.out_dtype == CSA_BF16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + row * dim;
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = threadIdx.x + u * kThreads;
      if (c < dim) o[c] = __float2bfloat16_rn(vals[u]);
    }
  } else {
    float* o = static_cast<float*>(a.out) + row * dim;
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u) {
      const int c = threadIdx.x + u * kThreads;
      if (c < dim) o[c] = vals[u];
    }
  }
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  dim3 grid(a.q_pos ? 1 : static_cast<unsigned>(a.n_ent), a.B);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  if (a.act_bf16)
    compress_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
  else
    compress_kernel<float><<<grid, kThreads, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
