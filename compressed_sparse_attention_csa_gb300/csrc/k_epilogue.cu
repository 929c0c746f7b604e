// Attention prologue / epilogue.
//
// "DeepSeek V4-Flash: The Cost of Deciding What to Read":
//  * "Grouped output projection": RMSNorm per head on the queries and on the single head of
//    the compressed KV entry, just before core attention;
//  * "Key and value are the same vector": RoPE on exactly the last 64 dims, and for a shared
//    key/value, RoPE at minus the query position on the last 64 dims of each head's output,
//    which vLLM fuses with the FP8 quantisation ahead of the output projection;
//  * vLLM also fuses the compressor with RMSNorm, RoPE and the cache insert.
// RoPE pairs are the interleaved (2j, 2j+1) of the rotated slice, angle pos * theta^(-2j/rd).
// An fp32 product pos * omega would be off by up to pos * 2^-24 rad (0.06 rad at 2^20), and
// double arithmetic runs at a small fraction of the fp32 rate on this part, so the phase is
// integer arithmetic: pos times the pair's 64-bit fixed-point turns per position, modulo 2^64;
// its top 32 bits give the angle in [-pi, pi) for the single-precision sine and cosine.
//
// All three are bandwidth- or latency-bound elementwise work: one warp per (row, head) vector
// for the norm / RoPE passes (16-byte loads, warp reductions), one CTA per entry for the
// compressor.
#include <cmath>

#include "csa_epi.h"
#include "csa_ptx.cuh"

namespace csa {
namespace {

constexpr float kLog2eF = 1.4426950408889634f;

__device__ __forceinline__ void rope_cs(int64_t pos, int j, const RopeTable& tab, float& c, float& s) {
  const uint64_t ph = static_cast<uint64_t>(pos) * tab.turn[j];             // turns, mod 1, as 2^-64 units
  const float ang = static_cast<float>(static_cast<int32_t>(ph >> 32)) * 1.4629180792671596e-9f;  // 2 pi / 2^32
  __sincosf(ang, &s, &c);
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Rotate the pairs of chunk `ch` (elements 8 ch .. 8 ch + 7) that fall in the last rd dims.
__device__ __forceinline__ void rope_chunk(float (&v)[8], int ch, int dim, int rd, int64_t pos, const RopeTable& tab) {
  const int r0 = dim - rd;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const int e = 8 * ch + i;
    if (e >= r0) {
      float c, s;
      rope_cs(pos, (e - r0) >> 1, tab, c, s);
      const float x0 = v[i], x1 = v[i + 1];
      v[i] = x0 * c - x1 * s;
      v[i + 1] = x0 * s + x1 * c;
    }
  }
}

constexpr int kVecWarps = 8;
constexpr int kVPW = 2;  // vectors a warp: the loads of both are issued before either is used

// ---- RMSNorm + RoPE, one warp per kVPW (row, head) vectors; CPL = 16-byte chunks a lane
template <typename T, int CPL>
__global__ void __launch_bounds__(32 * kVecWarps) norm_rope_kernel(const NormRopeArgs a) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t v0 = (static_cast<int64_t>(blockIdx.x) * kVecWarps + (threadIdx.x >> 5)) * kVPW;
  const int64_t nv = a.rows * a.heads;
  const int nch = a.dim >> 3;
  float x[kVPW][CPL][8];
#pragma unroll
  for (int u = 0; u < kVPW; ++u) {
    const int64_t v = v0 + u;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int ch = lane + 32 * q;
      if (v < nv && ch < nch) load8<T>(static_cast<const T*>(a.x) + v * a.dim + 8 * ch, x[u][q]);
    }
  }
#pragma unroll
  for (int u = 0; u < kVPW; ++u) {
    const int64_t v = v0 + u;
    if (v >= nv) break;
    const int64_t pos = a.pos[v / a.heads];
    float inv = 1.f;
    if (a.nr.weight) {
      float sq = 0.f;
#pragma unroll
      for (int q = 0; q < CPL; ++q)
        if (lane + 32 * q < nch) {
#pragma unroll
          for (int i = 0; i < 8; ++i) sq = fmaf(x[u][q][i], x[u][q][i], sq);
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      inv = 1.f / sqrtf(sq / static_cast<float>(a.dim) + a.nr.eps);
    }
    T* dst = static_cast<T*>(a.y) + v * a.dim;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int ch = lane + 32 * q;
      if (ch < nch) {
        if (a.nr.weight) {
          const float4 w0 = reinterpret_cast<const float4*>(a.nr.weight + 8 * ch)[0];
          const float4 w1 = reinterpret_cast<const float4*>(a.nr.weight + 8 * ch)[1];
          const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) x[u][q][i] = x[u][q][i] * inv * w[i];
        }
        if (a.nr.rope_dims > 0) rope_chunk(x[u][q], ch, a.dim, a.nr.rope_dims, pos, a.nr.tab);
        store8<T>(dst + 8 * ch, x[u][q]);
      }
    }
  }
}

// ---- inverse RoPE at -pos (+ e4m3 with one scale a vector), one warp per kVPW vectors
template <typename T, int CPL>
__global__ void __launch_bounds__(32 * kVecWarps) inv_rope_quant_kernel(const InvRopeArgs a) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t v0 = (static_cast<int64_t>(blockIdx.x) * kVecWarps + (threadIdx.x >> 5)) * kVPW;
  const int64_t nv = a.rows * a.heads;
  const int nch = a.dim >> 3;
  float x[kVPW][CPL][8];
#pragma unroll
  for (int u = 0; u < kVPW; ++u) {
    const int64_t v = v0 + u;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int ch = lane + 32 * q;
      if (v < nv && ch < nch) load8<T>(static_cast<const T*>(a.o) + v * a.dim + 8 * ch, x[u][q]);
    }
  }
#pragma unroll
  for (int u = 0; u < kVPW; ++u) {
    const int64_t v = v0 + u;
    if (v >= nv) break;
    const int64_t pos = -a.pos[v / a.heads];
    float am = 0.f;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int ch = lane + 32 * q;
      if (ch < nch) {
        if (a.rope_dims > 0) rope_chunk(x[u][q], ch, a.dim, a.rope_dims, pos, a.tab);
#pragma unroll
        for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(x[u][q][i]));
      }
    }
    if (!a.e4m3) {
      T* dst = static_cast<T*>(a.out) + v * a.dim;
#pragma unroll
      for (int q = 0; q < CPL; ++q) {
        const int ch = lane + 32 * q;
        if (ch < nch) store8<T>(dst + 8 * ch, x[u][q]);
      }
      continue;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float scale = am > 0.f ? __fdiv_rn(am, 448.f) : 1.f;
    uint8_t* dst = static_cast<uint8_t*>(a.out) + v * a.dim;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
      const int ch = lane + 32 * q;
      if (ch < nch) {
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i >> 2] |= static_cast<uint32_t>(f_to_e4m3(__fdiv_rn(x[u][q][i], scale))) << (8 * (i & 3));
        *reinterpret_cast<uint2*>(dst + 8 * ch) = make_uint2(w[0], w[1]);
      }
    }
    if (lane == 0) a.out_scale[v] = scale;
  }
}

// ---- compressor + RMSNorm + RoPE + cache insert, one CTA per (entry, sequence)
// Thread (slice s, pair p) takes channels 2p, 2p+1: all 2m tokens of the two-stream entry
// (S = 1), or tokens s, s + S, ... of the one-stream block; batches of 16 tokens' loads in
// flight, batch maximum, independent weights; slices merged in shared memory; then the
// entry's mean square (block reduction), the RMSNorm weight, and RoPE at position m * i.
template <typename T, bool TWO>
__global__ void __launch_bounds__(512) compress_norm_rope_kernel(const CompressEpiArgs a, int S) {
  extern __shared__ float s_epi[];  // [S][3][dim] slice partials, then [32] warp sums
  pdl_wait();
  pdl_trigger();
  const int np = a.dim >> 1;
  const int tid = threadIdx.x, p = tid % np, sl = tid / np;
  const int c = 2 * p;
  const int b = blockIdx.y;
  const int64_t entry = a.ent_begin + blockIdx.x;
  const int m = a.m;
  const T* kv = static_cast<const T*>(a.kv);
  const T* z = static_cast<const T*>(a.z);
  float mx0 = -INFINITY, mx1 = -INFINITY, sm0 = 0.f, sm1 = 0.f, ac0 = 0.f, ac1 = 0.f;
  // token u of this thread -> (element offset of its (C, Z) pair, bias offset)
  const int n_tk = TWO ? (entry > 0 ? 2 * m : m) : (m - sl + S - 1) / S;
  for (int u0 = 0; u0 < n_tk; u0 += 16) {
    // every load of the batch first (tokens past the list read its first token and are
    // dropped below), so that they are in flight together; the bias is added after
    float2 lg[16], val[16], bb[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int u = u0 + q < n_tk ? u0 + q : 0;
      int64_t off;
      int64_t boff;
      if (TWO) {
        const int st = u < m ? 0 : 1, j = u < m ? u : u - m;
        const int64_t row = (st == 0 ? m * entry : m * (entry - 1)) + j - a.tok0;
        off = ((static_cast<int64_t>(b) * a.n_tok + row) * 2 + st) * a.dim + c;
        boff = static_cast<int64_t>(st * m + j) * a.dim + c;
      } else {
        const int j = sl + S * u;
        const int64_t row = m * entry + j - a.tok0;
        off = (static_cast<int64_t>(b) * a.n_tok + row) * a.dim + c;
        boff = static_cast<int64_t>(j) * a.dim + c;
      }
      if constexpr (sizeof(T) == 2) {
        lg[q] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(z + off));
        val[q] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kv + off));
      } else {
        lg[q] = *reinterpret_cast<const float2*>(z + off);
        val[q] = *reinterpret_cast<const float2*>(kv + off);
      }
      bb[q] = a.bias ? *reinterpret_cast<const float2*>(a.bias + boff) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (u0 + q < n_tk) {
        lg[q].x += bb[q].x;
        lg[q].y += bb[q].y;
      } else {
        lg[q] = make_float2(-INFINITY, -INFINITY);
        val[q] = make_float2(0.f, 0.f);
      }
    }
    float b0 = mx0, b1 = mx1;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      b0 = fmaxf(b0, lg[q].x);
      b1 = fmaxf(b1, lg[q].y);
    }
    const float r0 = mx0 == -INFINITY ? 0.f : exp2f((mx0 - b0) * kLog2eF);
    const float r1 = mx1 == -INFINITY ? 0.f : exp2f((mx1 - b1) * kLog2eF);
    sm0 *= r0; ac0 *= r0; sm1 *= r1; ac1 *= r1;
    mx0 = b0;
    mx1 = b1;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float e0 = exp2f((lg[q].x - b0) * kLog2eF), e1 = exp2f((lg[q].y - b1) * kLog2eF);
      sm0 += e0;
      sm1 += e1;
      ac0 = fmaf(e0, val[q].x, ac0);
      ac1 = fmaf(e1, val[q].y, ac1);
    }
  }
  float v0 = 0.f, v1 = 0.f;
  if (S > 1) {
    float* r = s_epi + static_cast<int64_t>(sl) * 3 * a.dim;
    r[c] = mx0; r[c + 1] = mx1;
    r[a.dim + c] = sm0; r[a.dim + c + 1] = sm1;
    r[2 * a.dim + c] = ac0; r[2 * a.dim + c + 1] = ac1;
    __syncthreads();
    if (sl == 0) {
      float res[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float M = -INFINITY;
        for (int q = 0; q < S; ++q) M = fmaxf(M, s_epi[q * 3 * a.dim + c + k]);
        float sum = 0.f, acc = 0.f;
        for (int q = 0; q < S; ++q) {
          const float ms = s_epi[q * 3 * a.dim + c + k];
          if (ms != -INFINITY) {
            const float f = exp2f((ms - M) * kLog2eF);
            sum = fmaf(s_epi[q * 3 * a.dim + a.dim + c + k], f, sum);
            acc = fmaf(s_epi[q * 3 * a.dim + 2 * a.dim + c + k], f, acc);
          }
        }
        res[k] = acc / sum;
      }
      v0 = res[0];
      v1 = res[1];
    }
  } else {
    v0 = ac0 / sm0;
    v1 = ac1 / sm1;
  }
  // the entry's mean square over its dim channels (threads of slice 0 hold them)
  float sq = sl == 0 ? v0 * v0 + v1 * v1 : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  float* s_sq = s_epi + static_cast<int64_t>(S) * 3 * a.dim;
  __syncthreads();  // the slice partials have been read
  if ((tid & 31) == 0) s_sq[tid >> 5] = sq;
  __syncthreads();
  if (sl != 0) return;
  float tot = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += s_sq[w];
  if (a.nr.weight) {
    const float inv = 1.f / sqrtf(tot / static_cast<float>(a.dim) + a.nr.eps);
    const float2 w = *reinterpret_cast<const float2*>(a.nr.weight + c);
    v0 = v0 * inv * w.x;
    v1 = v1 * inv * w.y;
  }
  const int r0 = a.dim - a.nr.rope_dims;
  if (a.nr.rope_dims > 0 && c >= r0) {
    float cs, sn;
    rope_cs(static_cast<int64_t>(m) * entry, (c - r0) >> 1, a.nr.tab, cs, sn);
    const float x0 = v0, x1 = v1;
    v0 = x0 * cs - x1 * sn;
    v1 = x0 * sn + x1 * cs;
  }
  const int64_t row = static_cast<int64_t>(b) * a.E_cap + entry;
  if (a.fp8kv) {  // FP8 main-KV entry: e4m3 codes of dims < dim - 64, then bf16
    uint8_t* o = static_cast<uint8_t*>(a.out) + row * (a.dim + 64);
    const int nf = a.dim - 64;
    if (c < nf) {
      *reinterpret_cast<uint16_t*>(o + c) =
          static_cast<uint16_t>(f_to_e4m3(v0) | (static_cast<uint16_t>(f_to_e4m3(v1)) << 8));
    } else {
      *reinterpret_cast<__nv_bfloat162*>(o + nf + 2 * (c - nf)) = __floats2bfloat162_rn(v0, v1);
    }
    return;
  }
  if constexpr (sizeof(T) == 2)
    *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(a.out) + row * a.dim + c) =
        __floats2bfloat162_rn(v0, v1);
  else
    *reinterpret_cast<float2*>(static_cast<float*>(a.out) + row * a.dim + c) = make_float2(v0, v1);
}

// ---- pack rows into FP8 main-KV entries, one warp per row
template <typename T, int CPL>
__global__ void __launch_bounds__(32 * kVecWarps) kv_pack_fp8_kernel(const KvPackArgs a) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kVecWarps + (threadIdx.x >> 5);
  if (r >= a.rows) return;
  const int nch = a.dim >> 3, nf = a.dim - 64;
  float x[CPL][8];
#pragma unroll
  for (int q = 0; q < CPL; ++q) {
    const int ch = lane + 32 * q;
    if (ch < nch) load8<T>(static_cast<const T*>(a.x) + r * a.dim + 8 * ch, x[q]);
  }
  uint8_t* o = static_cast<uint8_t*>(a.out) + r * (a.dim + 64);
#pragma unroll
  for (int q = 0; q < CPL; ++q) {
    const int ch = lane + 32 * q;
    if (ch >= nch) continue;
    if (8 * ch < nf) {
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i >> 2] |= static_cast<uint32_t>(f_to_e4m3(x[q][i])) << (8 * (i & 3));
      *reinterpret_cast<uint2*>(o + 8 * ch) = make_uint2(w[0], w[1]);
    } else {
      store8<__nv_bfloat16>(reinterpret_cast<__nv_bfloat16*>(o + nf + 2 * (8 * ch - nf)), x[q]);
    }
  }
}

// ---- pack rows into MXFP4 entries: one warp a row, lane = a block of 16 channels
template <typename T>
__global__ void __launch_bounds__(32 * kVecWarps) kv_pack_mxfp4_kernel(const KvPackArgs a) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kVecWarps + (threadIdx.x >> 5);
  if (r >= a.rows) return;
  const int nb = a.dim >> 4;
  uint8_t* o = static_cast<uint8_t*>(a.out) + r * (a.dim / 2 + nb);
  for (int blk = lane; blk < nb; blk += 32) {
    float x[16];
    load8<T>(static_cast<const T*>(a.x) + r * a.dim + 16 * blk, *reinterpret_cast<float(*)[8]>(x));
    load8<T>(static_cast<const T*>(a.x) + r * a.dim + 16 * blk + 8, *reinterpret_cast<float(*)[8]>(x + 8));
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(x[i]));
    const uint8_t sc_code = f_to_e4m3(__fdiv_rn(am, 6.f));
    const float sc = e4m3_to_f(sc_code);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t c = sc > 0.f ? e2m1_code(__fdiv_rn(x[i], sc)) : 0u;
      w[i >> 3] |= c << (4 * (i & 7));
    }
    *reinterpret_cast<uint2*>(o + 8 * blk) = make_uint2(w[0], w[1]);
    o[a.dim / 2 + blk] = sc_code;
  }
}

}  // namespace

cudaError_t launch_kv_pack_mxfp4(const KvPackArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((a.rows + kVecWarps - 1) / kVecWarps));
  const dim3 blk(32 * kVecWarps);
  const cudaError_t e = a.bf16 ? launch_pdl(kv_pack_mxfp4_kernel<__nv_bfloat16>, grid, blk, 0, s, a)
                               : launch_pdl(kv_pack_mxfp4_kernel<float>, grid, blk, 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_kv_pack_fp8(const KvPackArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((a.rows + kVecWarps - 1) / kVecWarps));
  const dim3 blk(32 * kVecWarps);
  const bool two = a.dim <= 512;
  cudaError_t e;
  if (a.bf16)
    e = two ? launch_pdl(kv_pack_fp8_kernel<__nv_bfloat16, 2>, grid, blk, 0, s, a)
            : launch_pdl(kv_pack_fp8_kernel<__nv_bfloat16, 4>, grid, blk, 0, s, a);
  else
    e = two ? launch_pdl(kv_pack_fp8_kernel<float, 2>, grid, blk, 0, s, a)
            : launch_pdl(kv_pack_fp8_kernel<float, 4>, grid, blk, 0, s, a);
  count_launches(1);
  return e;
}

void make_rope_table(float theta, int rope_dims, RopeTable* t) {
  *t = RopeTable{};
  const long double two_pi = 6.283185307179586476925286766559005768L;
  const long double two64 = 18446744073709551616.0L;
  for (int j = 0; j < rope_dims / 2 && j < kMaxRopeDims / 2; ++j) {
    const long double w = std::pow(static_cast<long double>(theta), -2.0L * j / rope_dims);
    t->turn[j] = static_cast<uint64_t>(std::floor(w / two_pi * two64 + 0.5L));
  }
}

cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s) {
  const int64_t n = a.rows * a.heads;
  if (n == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((n + kVecWarps * kVPW - 1) / (kVecWarps * kVPW)));
  const dim3 blk(32 * kVecWarps);
  const bool two = a.dim <= 512;  // chunks a lane: 2 (dim <= 512) or 4 (dim <= 1024)
  cudaError_t e;
  if (a.bf16)
    e = two ? launch_pdl(norm_rope_kernel<__nv_bfloat16, 2>, grid, blk, 0, s, a)
            : launch_pdl(norm_rope_kernel<__nv_bfloat16, 4>, grid, blk, 0, s, a);
  else
    e = two ? launch_pdl(norm_rope_kernel<float, 2>, grid, blk, 0, s, a)
            : launch_pdl(norm_rope_kernel<float, 4>, grid, blk, 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_inv_rope_quant(const InvRopeArgs& a, cudaStream_t s) {
  const int64_t n = a.rows * a.heads;
  if (n == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((n + kVecWarps * kVPW - 1) / (kVecWarps * kVPW)));
  const dim3 blk(32 * kVecWarps);
  const bool two = a.dim <= 512;
  cudaError_t e;
  if (a.bf16)
    e = two ? launch_pdl(inv_rope_quant_kernel<__nv_bfloat16, 2>, grid, blk, 0, s, a)
            : launch_pdl(inv_rope_quant_kernel<__nv_bfloat16, 4>, grid, blk, 0, s, a);
  else
    e = two ? launch_pdl(inv_rope_quant_kernel<float, 2>, grid, blk, 0, s, a)
            : launch_pdl(inv_rope_quant_kernel<float, 4>, grid, blk, 0, s, a);
  count_launches(1);
  return e;
}

cudaError_t launch_compress_norm_rope(const CompressEpiArgs& a, cudaStream_t s) {
  if (a.n_ent == 0 || a.B == 0) return cudaSuccess;
  const int np = a.dim / 2;
  int S = 1;
  if (!a.two_stream) {
    S = 512 / np;
    if (S > 4) S = 4;
    if (S > a.m) S = a.m;
    if (S < 1) S = 1;
  }
  const dim3 grid(static_cast<unsigned>(a.n_ent), static_cast<unsigned>(a.B));
  const size_t smem = static_cast<size_t>(S) * 3 * a.dim * 4 + 32 * 4;
  cudaError_t e;
  if (a.two_stream)
    e = a.bf16 ? launch_pdl(compress_norm_rope_kernel<__nv_bfloat16, true>, grid, dim3(np * S), smem, s, a, S)
               : launch_pdl(compress_norm_rope_kernel<float, true>, grid, dim3(np * S), smem, s, a, S);
  else
    e = a.bf16 ? launch_pdl(compress_norm_rope_kernel<__nv_bfloat16, false>, grid, dim3(np * S), smem, s, a, S)
               : launch_pdl(compress_norm_rope_kernel<float, false>, grid, dim3(np * S), smem, s, a, S);
  count_launches(1);
  return e;
}

}  // namespace csa
