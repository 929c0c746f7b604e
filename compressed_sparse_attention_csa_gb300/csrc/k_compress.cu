// Gated two-stream KV compression.
//
// "DeepSeek V4-Flash: The Cost of Deciding What to Read", section "The compressor has two
// streams and they overlap": compressed entry i draws stream a (C^a, gate Z^a) from tokens
// [m*i, m*(i+1)) and stream b (C^b, Z^b) from [m*(i-1), m*i); a softmax over those 2m
// gate logits, with the learnable positional bias B^a / B^b added by position inside the
// block, runs independently for every channel, and the entry is the weighted sum of the
// matching C values.  Entry 0 has no previous block and mixes the m stream-a tokens only.
//
// Bandwidth/latency-bound: one CTA per (entry, sequence, job) where a job is one cache (main
// KV or indexer keys, both in one launch); one thread per channel; the 2m gate and value
// loads of a channel are issued before any arithmetic.  fp32 math; an E4M3 output gets one
// fp32 scale per entry (amax/448, codes rounded to nearest, saturating).
#include "csa_internal.h"
#include "csa_ptx.cuh"

namespace csa {
namespace {

constexpr int kMaxTok = 32;  // 2m <= 32

template <typename T>
__global__ void __launch_bounds__(512) compress_kernel(CompressArgs a) {
  pdl_wait();  // the caches and histograms may still be read by the previous step
  pdl_trigger();
  const CompressJob& job = a.job[blockIdx.z];
  const int b = blockIdx.y;
  const int m = a.m;
  if (a.zero_hist && blockIdx.x == 0 && blockIdx.z == 0) {
    for (int i = threadIdx.x; i < kTopkHistRowWords; i += blockDim.x)
      a.zero_hist[static_cast<int64_t>(b) * kTopkHistRowWords + i] = 0u;
    if (threadIdx.x == 0) a.zero_hist[static_cast<int64_t>(a.B) * kTopkHistRowWords + b] = 0u;
  }
  int64_t entry, tok0, n_tok;
  if (a.q_pos) {
    const int64_t t = a.q_pos[b];
    if ((t + 1) % m != 0) return;
    entry = (t + 1) / m - 1;
    tok0 = t - 2 * m + 1;
    n_tok = 2 * m;
  } else {
    entry = a.ent_begin + blockIdx.x;
    tok0 = a.tok0;
    n_tok = a.n_tok;
  }
  if (entry < 0 || entry >= a.E_cap) return;
  const int dim = job.dim;
  const int c = threadIdx.x;
  const T* kv = static_cast<const T*>(job.kv) + static_cast<int64_t>(b) * n_tok * 2 * dim;
  const T* z = static_cast<const T*>(job.z) + static_cast<int64_t>(b) * n_tok * 2 * dim;
  const int nt = entry == 0 ? m : 2 * m;  // stream-a tokens first, then stream-b tokens

  float v = 0.f;
  if (c < dim) {
    float lg[kMaxTok], val[kMaxTok];
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      if (j < nt) {
        const int st = j < m ? 0 : 1;
        const int jj = j < m ? j : j - m;
        const int64_t tok = (st == 0 ? m * entry : m * (entry - 1)) + jj;
        const int64_t off = ((tok - tok0) * 2 + st) * dim + c;
        lg[j] = load_f<T>(z + off) + job.bias[(st * m + jj) * dim + c];
        val[j] = load_f<T>(kv + off);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j)
      if (j < nt) mx = fmaxf(mx, lg[j]);
    float sum = 0.f, acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      if (j < nt) {
        const float e = expf(lg[j] - mx);
        sum += e;
        acc = fmaf(e, val[j], acc);
      }
    }
    v = acc / sum;
  }

  const int64_t row = static_cast<int64_t>(b) * a.E_cap + entry;
  if (job.out_dtype == CSA_E4M3) {
    __shared__ float s_red[16];
    float am = c < dim ? fabsf(v) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = am;
    __syncthreads();
    am = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) am = fmaxf(am, s_red[w]);
    const float scale = am > 0.f ? __fdiv_rn(am, 448.f) : 1.f;
    if (c < dim) static_cast<uint8_t*>(job.out)[row * dim + c] = f_to_e4m3(__fdiv_rn(v, scale));
    if (threadIdx.x == 0) job.out_scale[row] = scale;
  } else if (c < dim) {
    if (job.out_dtype == CSA_BF16)
      static_cast<__nv_bfloat16*>(job.out)[row * dim + c] = __float2bfloat16_rn(v);
    else
      static_cast<float*>(job.out)[row * dim + c] = v;
  }
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  dim3 grid(a.q_pos ? 1 : static_cast<unsigned>(a.n_ent), a.B, a.n_jobs);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  int dmax = a.job[0].dim;
  if (a.n_jobs > 1 && a.job[1].dim > dmax) dmax = a.job[1].dim;
  const int threads = (dmax + 31) / 32 * 32;
  const cudaError_t e = a.act_bf16 ? launch_pdl(compress_kernel<__nv_bfloat16>, grid, dim3(threads), 0, s, a)
                                   : launch_pdl(compress_kernel<float>, grid, dim3(threads), 0, s, a);
  count_launches(1);
  return e;
}

}  // namespace csa
