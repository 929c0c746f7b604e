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
// fp32 scale per entry (amax/448, codes rounded to nearest, saturating); an MXFP4 output (the
// indexer keys, dim 128) one UE8M0 scale per 32 channels (a warp: the OCP MX rule
// 2^(floor(log2 amax) - 2)) and E2M1 codes, two to a byte.  In the decode step
// the same launch carries extra CTAs that write the indexer's query images (qprep_dev.cuh).
#include "csa_internal.h"
#include "csa_ptx.cuh"
#include "qprep_dev.cuh"

namespace csa {
namespace {

constexpr int kMaxTok = 32;  // 2m <= 32

template <typename T>
__global__ void __launch_bounds__(512) compress_kernel(CompressArgs a, QprepPart qp) {
  pdl_wait();  // the caches, images and histograms may still be read by the previous step
  pdl_trigger();
  const int b = blockIdx.y;
  if (static_cast<int>(blockIdx.z) >= a.n_jobs) {
    // decode step: the indexer's query images, one (query, head) row per warp
    const int nw = static_cast<int>(blockDim.x >> 5);
    const int gh = (static_cast<int>(blockIdx.z) - a.n_jobs) * nw + static_cast<int>(threadIdx.x >> 5);
    if (gh < qp.L.N) {
      if (qp.fp8)
        qprep_row<true>(qp.ia, qp.L, qprep_image(qp.L, qp.images, 0, b), 0, b, gh, threadIdx.x & 31);
      else
        qprep_row<false>(qp.ia, qp.L, qprep_image(qp.L, qp.images, 0, b), 0, b, gh, threadIdx.x & 31);
    }
    return;
  }
  const CompressJob& job = a.job[blockIdx.z];
  const int m = a.m;
  if (a.zero_hist && blockIdx.x == 0 && blockIdx.z == 0) {
    for (int i = threadIdx.x; i < kTopkHistRowWords; i += blockDim.x)
      a.zero_hist[static_cast<int64_t>(b) * kTopkHistRowWords + i] = 0u;
    if (threadIdx.x == 0) a.zero_hist[static_cast<int64_t>(a.B) * kTopkHistRowWords + b] = 0u;
  }
  // Stream rows of the two token blocks: stream a (current block) starts at row ra0, stream b
  // (previous block) at row rb0.  Decode mode: the buffer holds tokens t-2m+1..t, so the rows
  // are fixed (b: 0..m-1, a: m..2m-1) and every load is issued before q_pos is known.
  int64_t entry = 0, ra0, rb0, n_tok;
  bool b_ok;
  if (a.q_pos) {
    ra0 = m;
    rb0 = 0;
    n_tok = 2 * m;
    b_ok = true;
  } else {
    entry = a.ent_begin + blockIdx.x;
    ra0 = m * entry - a.tok0;
    rb0 = m * (entry - 1) - a.tok0;
    n_tok = a.n_tok;
    b_ok = entry > 0;
  }
  const int dim = job.dim;
  const int c = threadIdx.x;
  const T* kv = static_cast<const T*>(job.kv) + static_cast<int64_t>(b) * n_tok * 2 * dim;
  const T* z = static_cast<const T*>(job.z) + static_cast<int64_t>(b) * n_tok * 2 * dim;

  // every load first (tokens past the block read its first row and are dropped below), so
  // that they are in flight together; the bias is added once they have landed
  float lg[kMaxTok], val[kMaxTok], bs[kMaxTok];
  if (c < dim) {
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) {
      const bool in = j < 2 * m && (j < m || b_ok);
      const int st = in && j >= m ? 1 : 0;
      const int jj = !in ? 0 : (j < m ? j : j - m);
      const int64_t off = (((st == 0 ? ra0 : rb0) + jj) * 2 + st) * dim + c;
      lg[j] = load_f<T>(z + off);
      bs[j] = job.bias[(st * m + jj) * dim + c];
      val[j] = load_f<T>(kv + off);
    }
#pragma unroll
    for (int j = 0; j < kMaxTok; ++j) lg[j] += bs[j];
  }
  if (a.q_pos) {
    const int64_t t = a.q_pos[b];
    if ((t + 1) % m != 0) return;
    entry = (t + 1) / m - 1;
  }
  if (entry < 0 || entry >= a.E_cap) return;
  const int nt = entry == 0 ? m : 2 * m;  // stream-a tokens first, then stream-b tokens

  float v = 0.f;
  if (c < dim) {
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
    if (threadIdx.x == 0) static_cast<float*>(job.out_scale)[row] = scale;
  } else if (job.out_dtype == CSA_MXFP4) {
    // one warp = one block of 32 channels (dim is a multiple of 32; warps past dim hold none)
    float am = c < dim ? fabsf(v) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const uint32_t sb = mx_e2m1_scale_byte(am);
    const uint32_t code = e2m1_code(__fdiv_rn(v, ue8m0_value(sb)));
    const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);  // channel c + 1
    if (c < dim) {
      if ((c & 1) == 0) static_cast<uint8_t*>(job.out)[row * (dim / 2) + c / 2] = static_cast<uint8_t>(code | (hi << 4));
      if ((c & 31) == 0) static_cast<uint8_t*>(job.out_scale)[row * (dim / 32) + c / 32] = static_cast<uint8_t>(sb);
    }
  } else if (c < dim) {
    if (job.out_dtype == CSA_BF16)
      static_cast<__nv_bfloat16*>(job.out)[row * dim + c] = __float2bfloat16_rn(v);
    else
      static_cast<float*>(job.out)[row * dim + c] = v;
  }
}

cudaError_t launch_impl(const CompressArgs& a, const QprepPart& qp, int qp_ctas, cudaStream_t s) {
  dim3 grid(a.q_pos ? 1 : static_cast<unsigned>(a.n_ent), a.B, a.n_jobs + qp_ctas);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  int dmax = a.job[0].dim;
  if (a.n_jobs > 1 && a.job[1].dim > dmax) dmax = a.job[1].dim;
  int threads = (dmax + 31) / 32 * 32;
  if (qp_ctas > 0 && threads < 256) threads = 256;
  const cudaError_t e = a.act_bf16 ? launch_pdl(compress_kernel<__nv_bfloat16>, grid, dim3(threads), 0, s, a, qp)
                                   : launch_pdl(compress_kernel<float>, grid, dim3(threads), 0, s, a, qp);
  count_launches(1);
  return e;
}

// ------------------------------------------------------------------ one stream, no overlap
// "DeepSeek V4-Flash: The Cost of Deciding What to Read", section "Heavily Compressed
// Attention" (the same compressor at m' = 128 with one KV stream, so no overlap), and the
// V4.1 diagram's "Encoder groups compress pairs" (ratio 2, channel-wise softmax per pair,
// no positional embedding).  CTA = (entry, sequence, 64 channels); thread (slice s, lane l)
// takes channels 2l, 2l+1 of the chunk over the tokens j = s, s+16, ... of the block: the loads
// of a batch of up to 8 tokens are issued before the first use (a whole m' = 128 block in
// one round trip), the batch maximum is taken first and the weights 2^((z - max) log2 e) then
// computed independently (the running sums are rescaled once a batch); the sixteen slices are
// combined through shared memory.  Decode mode issues its loads before it reads the position.
constexpr int kC1Slices = 16, kC1Chan = 64, kC1Batch = 8;  // 8 x 16 = 128 tokens' loads in one batch
constexpr float kC1Log2e = 1.4426950408889634f;

template <typename T>
__device__ __forceinline__ float2 load_f2(const T* p);
template <>
__device__ __forceinline__ float2 load_f2<float>(const float* p) { return *reinterpret_cast<const float2*>(p); }
template <>
__device__ __forceinline__ float2 load_f2<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

template <typename T>
__global__ void __launch_bounds__(32 * kC1Slices) compress1_kernel(const Compress1Args a) {
  __shared__ float s_red[kC1Slices][3][kC1Chan];
  pdl_wait();  // the cache row may still be read by the previous step
  pdl_trigger();
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int c = blockIdx.z * kC1Chan + 2 * lane;
  const bool live = c < a.dim;
  const int m = a.m;
  // Stream rows of the block: decode mode holds tokens t-m+1 .. t in rows 0 .. m-1, so its
  // loads are issued before q_pos is read; otherwise entry ent_begin + blockIdx.x.
  int64_t entry = a.ent_begin + blockIdx.x, r0, n_tok;
  if (a.q_pos) {
    r0 = 0;
    n_tok = m;
  } else {
    r0 = static_cast<int64_t>(m) * entry - a.tok0;
    n_tok = a.n_tok;
  }
  const T* kv = static_cast<const T*>(a.kv) + (static_cast<int64_t>(b) * n_tok + r0) * a.dim + c;
  const T* z = static_cast<const T*>(a.z) + (static_cast<int64_t>(b) * n_tok + r0) * a.dim + c;
  float mx0 = -INFINITY, mx1 = -INFINITY, sm0 = 0.f, sm1 = 0.f, ac0 = 0.f, ac1 = 0.f;
  bool first = true;
  if (live) {
    for (int j0 = sl; j0 < m; j0 += kC1Batch * kC1Slices) {
      // every load of the batch first (rows past the block read its row 0 and are masked
      // after), so that they are in flight together
      float2 lg[kC1Batch], v[kC1Batch], bb[kC1Batch];
#pragma unroll
      for (int u = 0; u < kC1Batch; ++u) {
        const int j = j0 + u * kC1Slices;
        const int64_t jr = j < m ? j : 0;
        lg[u] = load_f2<T>(z + jr * a.dim);
        v[u] = load_f2<T>(kv + jr * a.dim);
        bb[u] = a.bias ? *reinterpret_cast<const float2*>(a.bias + jr * a.dim + c) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kC1Batch; ++u) {
        if (j0 + u * kC1Slices < m) {
          lg[u].x += bb[u].x;
          lg[u].y += bb[u].y;
        } else {
          lg[u] = make_float2(-INFINITY, -INFINITY);
          v[u] = make_float2(0.f, 0.f);
        }
      }
      if (first && a.q_pos) {  // decode: produce the entry only if the token completes it
        const int64_t t = a.q_pos[b];
        if ((t + 1) % m != 0) return;
        entry = (t + 1) / m - 1;
      }
      first = false;
      // the batch's maximum first, then its weights (independent of one another)
      float b0 = mx0, b1 = mx1;
#pragma unroll
      for (int u = 0; u < kC1Batch; ++u) {
        b0 = fmaxf(b0, lg[u].x);
        b1 = fmaxf(b1, lg[u].y);
      }
      const float q0 = mx0 == -INFINITY ? 0.f : exp2f((mx0 - b0) * kC1Log2e);
      const float q1 = mx1 == -INFINITY ? 0.f : exp2f((mx1 - b1) * kC1Log2e);
      sm0 *= q0;
      ac0 *= q0;
      sm1 *= q1;
      ac1 *= q1;
      mx0 = b0;
      mx1 = b1;
#pragma unroll
      for (int u = 0; u < kC1Batch; ++u) {
        const float e0 = exp2f((lg[u].x - b0) * kC1Log2e), e1 = exp2f((lg[u].y - b1) * kC1Log2e);
        sm0 += e0;
        sm1 += e1;
        ac0 = fmaf(e0, v[u].x, ac0);
        ac1 = fmaf(e1, v[u].y, ac1);
      }
    }
  }
  if (a.q_pos && (!live || sl >= m)) {  // threads that loaded nothing still take the decision
    const int64_t t = a.q_pos[b];
    if ((t + 1) % m != 0) return;
    entry = (t + 1) / m - 1;
  }
  if (entry < 0 || entry >= a.E_cap) return;
  s_red[sl][0][2 * lane] = mx0;
  s_red[sl][0][2 * lane + 1] = mx1;
  s_red[sl][1][2 * lane] = sm0;
  s_red[sl][1][2 * lane + 1] = sm1;
  s_red[sl][2][2 * lane] = ac0;
  s_red[sl][2][2 * lane + 1] = ac1;
  __syncthreads();
  // the slices combined by warps 0 and 1: warp q takes channel 2 lane + q
  if (sl > 1 || !live) return;
  const int q = sl;
  float res;
  {
    const int cc = 2 * lane + q;
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kC1Slices; ++s) M = fmaxf(M, s_red[s][0][cc]);
    float sum = 0.f, acc = 0.f;
#pragma unroll
    for (int s = 0; s < kC1Slices; ++s) {
      const float ms = s_red[s][0][cc];
      if (ms != -INFINITY) {  // slices with no token of this block hold nothing
        const float f = exp2f((ms - M) * kC1Log2e);
        sum = fmaf(s_red[s][1][cc], f, sum);
        acc = fmaf(s_red[s][2][cc], f, acc);
      }
    }
    res = acc / sum;
  }
  const int64_t row = static_cast<int64_t>(b) * a.E_cap + entry;
  if (a.act_bf16)
    static_cast<__nv_bfloat16*>(a.out)[row * a.dim + c + q] = __float2bfloat16_rn(res);
  else
    static_cast<float*>(a.out)[row * a.dim + c + q] = res;
}

}  // namespace

cudaError_t launch_compress1(const Compress1Args& a, cudaStream_t s) {
  dim3 grid(a.q_pos ? 1u : static_cast<unsigned>(a.n_ent), static_cast<unsigned>(a.B),
            static_cast<unsigned>((a.dim + kC1Chan - 1) / kC1Chan));
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  const cudaError_t e = a.act_bf16 ? launch_pdl(compress1_kernel<__nv_bfloat16>, grid, dim3(32 * kC1Slices), 0, s, a)
                                   : launch_pdl(compress1_kernel<float>, grid, dim3(32 * kC1Slices), 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  QprepPart none{};
  return launch_impl(a, none, 0, s);
}

cudaError_t launch_compress_with_qprep(const CompressArgs& a, const QprepPart& q, cudaStream_t s) {
  if (!a.q_pos || q.L.n_qgroups != 1) return cudaErrorInvalidValue;  // decode step only (T = 1)
  int dmax = a.job[0].dim;
  if (a.n_jobs > 1 && a.job[1].dim > dmax) dmax = a.job[1].dim;
  int threads = (dmax + 31) / 32 * 32;
  if (threads < 256) threads = 256;
  const int nw = threads / 32;
  return launch_impl(a, q, (q.L.N + nw - 1) / nw, s);
}

}  // namespace csa
