// Attention prologue / epilogue kernels: RMSNorm, partial RoPE, inverse RoPE and FP8
// quantisation of the output, and the compressor fused with RMSNorm + RoPE + cache insert.
#pragma once
#include "csa_internal.h"

namespace csa {

constexpr int kMaxRopeDims = 128;

// Pair j of the rotated slice turns by pos * f_j of a full turn, f_j = theta^(-2j/rd) / (2 pi),
// held as the 64-bit fixed-point fraction turn[j] = f_j * 2^64 (formed on the host in extended
// precision): (pos * turn[j]) mod 2^64 is the exact phase to within pos * 2^-63 turns.
struct RopeTable {
  uint64_t turn[kMaxRopeDims / 2];
};

struct NormRope {
  const float* weight;  // [dim] RMSNorm weight, or null: no RMSNorm
  float eps;
  int rope_dims;        // rotary dims at the end of each head (even, 0 = none, <= kMaxRopeDims)
  float theta;          // rotary base
  RopeTable tab;
};
void make_rope_table(float theta, int rope_dims, RopeTable* t);

// x, y: [rows, heads, dim] (dim % 8 == 0, <= 1024); y may alias x.
struct NormRopeArgs {
  const void* x;
  void* y;
  int64_t rows;
  int heads, dim;
  const int64_t* pos;   // [rows]
  bool bf16;
  NormRope nr;
};
cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s);

// Compressor (two streams with overlap, or one stream without) fused with RMSNorm + RoPE of
// the entry (position m * i) and the store into the cache.
struct CompressEpiArgs {
  bool two_stream;
  const void* kv;       // two streams: [B, n_tok, 2, dim]; one stream: [B, n_tok, dim]
  const void* z;
  const float* bias;    // [2, m, dim] / [m, dim] or null (one stream)
  int B, m, dim;        // dim even, <= 1024
  int64_t n_tok, tok0, ent_begin, n_ent, E_cap;
  void* out;            // [B, E_cap, dim], or [B, E_cap, dim + 64] bytes with fp8kv
  bool bf16;
  bool fp8kv;           // store the entry as an FP8 main-KV entry
  NormRope nr;
};
cudaError_t launch_compress_norm_rope(const CompressEpiArgs& a, cudaStream_t s);

// Inverse RoPE at position -pos[row] on the last rope_dims dims of every head of o, written
// in the activation dtype or as e4m3 codes with one fp32 scale per (row, head).
struct InvRopeArgs {
  const void* o;        // [rows, heads, dim]
  int64_t rows;
  int heads, dim;
  const int64_t* pos;
  int rope_dims;
  float theta;
  RopeTable tab;
  bool bf16;
  void* out;
  bool e4m3;
  float* out_scale;     // [rows, heads] when e4m3
};
cudaError_t launch_inv_rope_quant(const InvRopeArgs& a, cudaStream_t s);

// FP8 main-KV entries (d - 64 e4m3 codes, then the last 64 dims in bf16: 576 B for d = 512).
// Pack rows [rows, d] (bf16 / fp32) into that format.
struct KvPackArgs {
  const void* x;
  void* out;            // [rows, d + 64] bytes
  int64_t rows;
  int dim;              // % 16 == 0, 64 < dim <= 1024
  bool bf16;
};
cudaError_t launch_kv_pack_fp8(const KvPackArgs& a, cudaStream_t s);

// Sparse attention over FP8 main-KV entries (kv_comp [B, E_cap, 576] bytes), decode shapes:
// the split plan of csa_sparse_attn's decode path (few queries, k + W > 128 rows).
bool attn_fp8kv_supported(int B, int T, int H, int d, int k, int W, int act, int num_sms);  // decode split plan
bool attn_quantkv_supported(int B, int T, int H, int d, int k, int W, int act, int num_sms);  // + many queries
cudaError_t launch_attn_fp8kv(const AttnArgs& a, cudaStream_t s);
// The same over MXFP4 main-KV entries (kv_comp [B, E_cap, 288] bytes).
cudaError_t launch_attn_mxfp4kv(const AttnArgs& a, cudaStream_t s);

// MXFP4 entries: per 16 channels one e4m3 scale = e4m3(amax / 6); codes = the nearest E2M1
// value of x / scale (ties to the even code, saturating, sign kept); element 2i in the low
// nibble; the dim/2 payload bytes, then the dim/16 scales.
cudaError_t launch_kv_pack_mxfp4(const KvPackArgs& a, cudaStream_t s);

}  // namespace csa
