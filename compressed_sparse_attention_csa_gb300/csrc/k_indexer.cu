// Lightning-indexer scores.
//
// "DeepSeek V4-Flash: The Cost of Deciding What to Read", section "The Lightning Indexer":
//   I(t, s) = sum_h w^I(t, h) * ReLU(q^I(t, h) . K^IComp_s)
// with 64 indexer heads of dimension 128 and one gate per head.  Causality ("The sliding
// window is not an optimisation"): a query at t reads entry s only if m(s+1) - 1 <= t, i.e.
// s < floor((t + 1) / m).  Every other column is -inf.
//
// Tensor-core path (bf16 or e4m3 keys, dI = 128): the contraction qI . kI is a dense GEMM
// with the KEYS as the M dimension: D[s, (g, h)] = kI[s] . qI[g, h] for a 128-key tile and
// the G*HI query-heads of a query group as N.  Each TMEM lane then holds one key's scores
// for every head, so ReLU, the gate weights and the sum over heads are thread-local in the
// epilogue.  Key tiles stream through a TMA ring (evict-first); one thread issues the MMAs
// into a ring of TMEM accumulators; two groups of four epilogue warps take alternate tiles.
// The query operand of each query group is prepared once (indexer_qprep_kernel) as the
// exact shared-memory image, and every CTA of the group pulls it with one bulk copy; with one
// query per sequence and the key range split over CTAs, each CTA builds the image itself.
//
// E4M3 keys use kind::f8f6f4.  The query is split into two E4M3 terms, q/s = hi + lo with
// s = per-head amax/448, and both terms run through the same accumulator (the K loop is
// issued twice, with the same key tile), so D = k . (hi + lo) to about bf16 accuracy.  The
// per-key fp32 scale and the per-head s are positive and factor out of the ReLU.
//
// MXFP4 keys ("FP4, down to the index scores"; 64 payload bytes + 4 UE8M0 scales a key) use
// the block-scaled kind::mxf8f6f4: A = E2M1 keys, B = the same two E4M3 query terms, and the
// keys' scales applied by the MMA from TMEM.  TMA unpacks the packed payload into the 8-bit
// slots the MMA reads (16 codes in each 16-byte chunk), so a key tile has the FP8 tile's
// shared-memory footprint at half its HBM bytes.  The MMA takes row r's scale from TMEM lane
// r, column (r / 32) of a 4-column group; a tile therefore holds key 4l + c (l = 0..31,
// c = 0..3) in row 32c + l, so that the tile's 128 scale words, contiguous in memory, are
// exactly the 32 lines of 16 bytes one tcgen05.cp (32x128b, copied to all four lane
// quadrants) puts in place.
#include <algorithm>
#include <type_traits>

#include "csa_internal.h"
#include "csa_ptx.cuh"
#include "qprep_dev.cuh"

namespace csa {
namespace {

// A score as the scores array holds it: fp32, or rounded to BF16 (nearest even) when the
// caller asked for BF16 scores; the histogram digit is taken from the stored value.
__device__ __forceinline__ float stored_score(const IndexerArgs& a, float v) {
  return a.scores_bf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}
__device__ __forceinline__ void store_score(const IndexerArgs& a, int64_t i, float v) {
  if (a.scores_bf16)
    reinterpret_cast<__nv_bfloat16*>(a.scores)[i] = __float2bfloat16_rn(v);
  else
    a.scores[i] = v;
}

// ------------------------------------------------------------------ CUDA-core path
struct MxKey {};  // key type tag: MXFP4 keys (DI/2 payload bytes and one scale word per key)

template <typename TQ, typename TK, int DI>
__global__ void __launch_bounds__(128) indexer_simt_kernel(IndexerArgs a, int64_t n_cols) {
  extern __shared__ float sm[];
  float* sq = sm;              // [HI][DI]
  float* sw = sm + a.HI * DI;  // [HI]
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.y;
  const int b = static_cast<int>(row / a.T);
  const TQ* q = static_cast<const TQ*>(a.qI) + row * a.HI * DI;
  for (int i = threadIdx.x; i < a.HI * DI; i += blockDim.x) sq[i] = load_f<TQ>(q + i);
  for (int i = threadIdx.x; i < a.HI; i += blockDim.x) sw[i] = a.w[row * a.HI + i];
  __syncthreads();
  const int64_t col = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (col >= n_cols) return;
  const int64_t t = a.q_pos[row];
  int64_t nv = t < 0 ? 0 : (t + 1) / a.m;
  nv = nv < a.E_cap ? nv : a.E_cap;
  if (a.nv_out && col == 0) a.nv_out[row] = static_cast<int32_t>(nv);
  const int64_t s = a.cand ? a.cand[row * a.n_cand + col] : col;
  float score = -INFINITY;
  if (s >= 0 && s < nv) {
    float kv[DI];
    const int64_t krow = static_cast<int64_t>(b) * a.E_cap + s;
    if constexpr (std::is_same<TK, MxKey>::value) {
      const uint8_t* kp = static_cast<const uint8_t*>(a.kI) + krow * (DI / 2);
      const uint32_t sw = static_cast<const uint32_t*>(a.kscale)[krow];
#pragma unroll
      for (int c = 0; c < DI; ++c)
        kv[c] = e2m1_value((kp[c >> 1] >> (4 * (c & 1))) & 15u) * ue8m0_value((sw >> (8 * (c >> 5))) & 0xFFu);
    } else if constexpr (std::is_same<TK, uint8_t>::value) {
      const uint8_t* kp = static_cast<const uint8_t*>(a.kI) + krow * DI;
#pragma unroll
      for (int c = 0; c < DI; ++c) kv[c] = e4m3_to_f(kp[c]);
    } else {
      const TK* kp = static_cast<const TK*>(a.kI) + krow * DI;
#pragma unroll
      for (int c = 0; c < DI; ++c) kv[c] = load_f<TK>(kp + c);
    }
    float acc = 0.f;
    for (int h = 0; h < a.HI; ++h) {
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < DI; ++c) dot = fmaf(sq[h * DI + c], kv[c], dot);
      acc = fmaf(sw[h], fmaxf(dot, 0.f), acc);
    }
    if constexpr (std::is_same<TK, uint8_t>::value) acc *= static_cast<const float*>(a.kscale)[krow];
    score = acc;
  }
  store_score(a, row * a.ld + col, score);
}

// ------------------------------------------------------------------ tensor-core path
// Warp 0 TMA, warp 1 MMA + TMEM, then the epilogue warps: 8 with two CTAs per SM, 16 with one.
constexpr int epi_warps(int minb) { return minb == 1 ? 16 : 8; }
constexpr int tc_threads(int minb) { return 64 + 32 * epi_warps(minb); }
constexpr int kTcThreads = tc_threads(2);
constexpr int kTile = 128;                       // keys per tile (MMA M)
constexpr int kMaxG = 8;
constexpr uint32_t kKeyTileBytesF8 = kTile * 128;  // 128 keys x 128 e4m3 codes (or unpacked E2M1)
// key formats of the tensor-core path
constexpr int kKeyBf16 = 0, kKeyE4m3 = 1, kKeyMx = 2;
constexpr uint32_t kMxScaleSlot = kTile * 4;       // a tile's 128 scale words
constexpr uint32_t kMxBoxBytes = 32 * 64;          // one TMA box: 32 keys x 64 packed bytes

using TcLayout = IndexerLayout;

// One query per sequence over dense keys (two CTAs per SM, the key range split): every CTA
// converts the query itself (16 KiB read from L2) instead of waiting for a query-prep launch.
__host__ __device__ __forceinline__ bool image_in_cta(const IndexerArgs& a, const TcLayout& L) {
  return !L.wide && a.T == 1 && a.cand == nullptr;
}

__device__ __forceinline__ bool wait_time_only(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitBudgetNs) return false;
  return true;
}


// sum_j w[j] * relu(v[j]) over 32 values (w in shared memory, read as float4), four chains
__device__ __forceinline__ float relu_dot32(const float (&v)[32], const float* w) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 w4 = *reinterpret_cast<const float4*>(w + j);
    a0 = fmaf(w4.x, fmaxf(v[j], 0.f), a0);
    a1 = fmaf(w4.y, fmaxf(v[j + 1], 0.f), a1);
    a2 = fmaf(w4.z, fmaxf(v[j + 2], 0.f), a2);
    a3 = fmaf(w4.w, fmaxf(v[j + 3], 0.f), a3);
  }
  return (a0 + a1) + (a2 + a3);
}

// Query operand of every query group, written once as the CTA's shared-memory image
// (qprep_row in qprep_dev.cuh).  Grid (query group, sequence, row block of 8): one warp per
// (query, head) row, so every row's load is in flight at once.
template <bool FP8>
__global__ void __launch_bounds__(256) indexer_qprep_kernel(const IndexerArgs a, const TcLayout L,
                                                            uint8_t* images) {
  pdl_wait();  // the images may still be read by the previous indexer launch
  pdl_trigger();
  const int gh = blockIdx.z * 8 + (threadIdx.x >> 5);
  if (gh < L.N)
    qprep_row<FP8>(a, L, qprep_image(L, images, blockIdx.x, blockIdx.y), blockIdx.x, blockIdx.y, gh, threadIdx.x & 31);
}

// Warp 0: TMA producer.  Warp 1: TMEM owner and MMA issuer (it also pulls the query image).
// Warps 2..: epilogue, in groups of four (one warp per TMEM lane quadrant).  Groups take
// alternate tiles; with 16 epilogue warps (one CTA per SM) the two groups of a tile parity
// split its queries between them, which doubles the warps that hide the TMEM and shared
// memory latencies of the reduction.
template <int KF, bool FUSE, int MINB>
__global__ void __launch_bounds__(tc_threads(MINB), MINB) indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                   const IndexerArgs a, const TcLayout L,
                                                                   const uint8_t* images, const int64_t n_cols) {
  constexpr bool FP8 = KF == kKeyE4m3;   // e4m3 keys with one fp32 scale each
  constexpr bool MX = KF == kKeyMx;      // MXFP4 keys, block-scaled MMA
  constexpr bool F8Q = KF != kKeyBf16;   // the query as two e4m3 terms (both 8-bit key formats)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  const int HI = a.HI, G = L.G, N = L.N, S = L.stages;
  uint8_t* sB = smem;
  float* sW = reinterpret_cast<float*>(smem + L.b_bytes);  // [G][HI], right after the B image
  uint8_t* sA = smem + L.b_bytes + align_up_dev(L.w_bytes, 1024);
  // MXFP4: each stage's 128 key scale words
  uint8_t* sSc = sA + static_cast<size_t>(S) * L.stage_bytes;
  int* sNv = reinterpret_cast<int*>(sSc + (MX ? static_cast<size_t>(S) * kMxScaleSlot : 0));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_align(reinterpret_cast<uint8_t*>(sNv + kMaxG), 8));
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;       // [4] accumulator ready for the epilogue
  uint64_t* tempty = bars + 2 * S + 4;  // [4] accumulator drained
  uint64_t* qbar = bars + 2 * S + 8;    // query image landed
  uint64_t* kbar = bars + 2 * S + 9;    // decode step: the new key entry is written
  uint64_t* sbar = bars + 2 * S + 10;   // MXFP4: the query side's scales are in TMEM
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(bars + 2 * S + 11);
  volatile int* sAbort = reinterpret_cast<volatile int*>(sTmem + 1);
  int64_t* sNew = reinterpret_cast<int64_t*>(sTmem + 2);     // decode step: new entry (-1: none)
  float* sNewScale = reinterpret_cast<float*>(sTmem + 5);
  float* sRed4 = reinterpret_cast<float*>(sTmem + 8);        // [4] decode step: key amax
  uint32_t* sHist = sTmem + 12;                               // [4096] when a histogram is kept (G == 1)
  constexpr bool fuse = FUSE;  // decode step: see DecodeFuse
  const bool img_cta = FUSE || image_in_cta(a, L);  // the epilogue warps write the query image
  const bool hist = (a.hist_out != nullptr || fuse) && G == 1;
  const int NA = L.n_acc;
  // MXFP4: TMEM columns after the accumulators: a 4-column scale group per accumulator (the
  // tile's key scales), then the query side's scales (8 columns, 2^0 in every byte), each
  // group 8-aligned
  const uint32_t sf0 = (static_cast<uint32_t>(NA * N) + 7u) & ~7u;
  const uint32_t sfb_col = sf0 + 8u * static_cast<uint32_t>(NA);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, qg = blockIdx.y, g0 = qg * G, split = blockIdx.x;
  const int T = a.T;
  const int64_t qrow0 = static_cast<int64_t>(b) * T + g0;

  constexpr int EPI = epi_warps(MINB);
  // epilogue groups per tile (two split the queries when there are 16 warps and >= 2 queries)
  const int gpt = (EPI == 16 && G >= 2) ? 2 : 1;
  if (hist)
    for (int i = tid; i < kTopkHistBins; i += tc_threads(MINB)) sHist[i] = 0u;
  if (tid < kMaxG) {
    int nv = 0;
    if (tid < G && g0 + tid < T) {
      const int64_t t = a.q_pos[qrow0 + tid];
      int64_t v = t < 0 ? 0 : (t + 1) / a.m;
      nv = static_cast<int>(v < a.E_cap ? v : a.E_cap);
      if (a.nv_out && split == 0) a.nv_out[qrow0 + tid] = nv;
      if (fuse && tid == 0) {
        // the entry the token completes (compressed in this launch), if it fits the cache
        const int64_t e = t >= 0 && (t + 1) % a.m == 0 ? (t + 1) / a.m - 1 : -1;
        *sNew = e < a.E_cap ? e : -1;
      }
    }
    sNv[tid] = nv;
  }
  if (tid == 0) *sAbort = 0;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], !FUSE && a.cand ? 32 : 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 32 * 4 * gpt);
    }
    mbar_init(qbar, img_cta ? 32 * EPI : 1);
    mbar_init(kbar, 1);
    mbar_init(sbar, 128);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sTmem, L.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  // the keys, scales, query images and histograms are written by the kernels before this one
  // (decode step: nothing this launch reads is written by earlier kernels of the step)
  if (!fuse) pdl_wait();
  const int64_t e_new = fuse ? *sNew : -1;

  int nv_max = 0;
  for (int g = 0; g < G; ++g) nv_max = max(nv_max, sNv[g]);
  if (!FUSE && a.cand) nv_max = a.n_cand;  // candidate slots, each checked against the visible count
  const int tiles_needed = (nv_max + kTile - 1) / kTile;
  // the splits of a row interleave tile by tile (split, split + n_splits, ...)
  const int tile_lo = split, tile_step = L.n_splits;
  const int n_it = tiles_needed > tile_lo ? (tiles_needed - tile_lo + tile_step - 1) / tile_step : 0;

  if (warp == 0) {
    // decode step: this CTA scores the tile of the new entry (its last tile), whose key the
    // epilogue warps compress first: that tile is loaded once the key is written
    const bool own_new =
        e_new >= 0 && n_it > 0 && static_cast<int64_t>(tile_lo + (n_it - 1) * tile_step) == e_new / kTile;
    const int key_it = own_new ? n_it - 1 : n_it;
    if (n_it > 0) {
      uint64_t pol = 0;
      bool ok = true;
      int issued = 0;
      const bool gather = !FUSE && !MX && a.cand != nullptr;  // the decode step has no candidate lists
      if (lane == 0 && !gather) {
        tma_prefetch_desc(&kmap);
        pol = policy_evict_first();
      }
      auto issue = [&](int it) {
        const int st = it % S;
        if (!mbar_wait_b(&empty[st], ((it / S) & 1) ^ 1, a.err, sAbort, a.wait_ns)) return false;
        const int64_t row64 =
            static_cast<int64_t>(b) * a.E_cap + static_cast<int64_t>(tile_lo + it * tile_step) * kTile;
        uint8_t* dst = sA + static_cast<size_t>(st) * L.stage_bytes;
        if constexpr (MX) {
          // four boxes of 32 keys each: box c takes keys 4l + c (l = 0..31) of the tile into
          // rows 32c + l; the tile's scale words follow in one bulk copy (the last tile of the
          // cache copies only the words that exist)
          const int64_t left = static_cast<int64_t>(a.B) * a.E_cap - row64;
          const uint32_t sc_bytes = left >= kTile ? kMxScaleSlot : static_cast<uint32_t>(left) * 4u;
          mbar_arrive_expect_tx(&full[st], 4 * kMxBoxBytes + sc_bytes);
          const int r4 = static_cast<int>(row64 / 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_load_3d_hint(dst + c * 4096, &kmap, &full[st], 0, c, r4, pol);
          bulk_g2s(sSc + static_cast<size_t>(st) * kMxScaleSlot, static_cast<const uint32_t*>(a.kscale) + row64,
                   sc_bytes, &full[st]);
          return true;
        }
        mbar_arrive_expect_tx(&full[st], L.stage_bytes);
        const int row = static_cast<int>(row64);
        // innermost coordinate 0 or 64 elements: always 16-byte aligned
        tma_load_2d_hint(dst, &kmap, &full[st], 0, row, pol);
        if constexpr (!FP8) tma_load_2d_hint(dst + 16384, &kmap, &full[st], 64, row, pol);
        return true;
      };
      if (gather) {
        // candidate mode: the warp gathers each tile's rows with 16-byte cp.async into the
        // swizzled stage; once a stage's copies have landed it is fenced for the tensor core
        // and its full barrier arrived on (up to S - 1 later stages stay in flight)
        const int row_bytes = FP8 ? 128 : 256;
        const uint8_t* kbase = static_cast<const uint8_t*>(a.kI) + static_cast<size_t>(b) * a.E_cap * row_bytes;
        const int32_t* cb = a.cand + static_cast<int64_t>(qrow0) * a.n_cand;
        // each lane's copies of tile j are complete: it fences them for the tensor core and
        // arrives (the full barriers count 32 arrivals in this mode)
        auto land = [&](int j) {
          fence_proxy_async_smem();
          mbar_arrive(&full[j % S]);
        };
        const int lag = min(S - 1, 3);  // tiles left in flight behind the newest
        auto wait_lag = [&]() {
          if (lag >= 3)
            asm volatile("cp.async.wait_group 3;" ::: "memory");
          else if (lag == 2)
            asm volatile("cp.async.wait_group 2;" ::: "memory");
          else
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        };
        for (int it = 0; ok && it < n_it; ++it) {
          const int st = it % S;
          if (lane == 0) ok = mbar_wait_b(&empty[st], ((it / S) & 1) ^ 1, a.err, sAbort, a.wait_ns);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          uint8_t* dst = sA + static_cast<size_t>(st) * L.stage_bytes;
          const int slot0 = (tile_lo + it * tile_step) * kTile;
#pragma unroll
          for (int rr = 0; rr < kTile / 32; ++rr) {
            const int r = rr * 32 + lane;
            const int slot = slot0 + r;
            int64_t p = slot < a.n_cand ? cb[slot] : 0;
            p = (p >= 0 && p < a.E_cap) ? p : 0;  // invisible or padded slots read row 0 (masked later)
            const uint8_t* src = kbase + p * row_bytes;
#pragma unroll
            for (int c = 0; c < row_bytes / 16; ++c)
              cp_async16(dst + (c >> 3) * 16384 + sw128(r, c & 7), src + c * 16);
          }
          asm volatile("cp.async.commit_group;" ::: "memory");
          ++issued;
          if (issued > lag) {
            wait_lag();
            land(it - lag);
          }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        for (int j = max(0, issued - lag); j < issued; ++j) land(j);
      } else if (lane == 0 && !a.skip_key_loads) {
        for (int it = 0; ok && it < key_it; ++it) ok = issue(it), issued += ok;
        if (FUSE && own_new && ok) ok = mbar_wait_b(kbar, 0, a.err, sAbort, a.wait_ns);
        for (int it = key_it; ok && it < n_it; ++it) ok = issue(it), issued += ok;
        // every load issued must have landed before the CTA may exit
        for (int it = max(0, issued - S); it < issued; ++it) wait_time_only(&full[it % S], (it / S) & 1);
      }
    }
    // columns past the last visible tile: -inf (written by the last split of the group)
    if (split == L.n_splits - 1) {
      for (int g = 0; g < G; ++g) {
        if (g0 + g >= T) break;
        const int64_t r0 = (qrow0 + g) * a.ld;
        for (int64_t c = static_cast<int64_t>(tiles_needed) * kTile + lane; c < n_cols; c += 32)
          store_score(a, r0 + c, -INFINITY);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // the group's query image (B operand + gates): one bulk copy, or (one query per
      // sequence) written by the epilogue warps
      if (!img_cta) {
        const uint8_t* img = images + (static_cast<size_t>(b) * L.n_qgroups + qg) * (L.b_bytes + L.w_bytes);
        mbar_arrive_expect_tx(qbar, L.b_bytes + L.w_bytes);
        bulk_g2s(sB, img, L.b_bytes, qbar);
        bulk_g2s(sW, img + L.b_bytes, L.w_bytes, qbar);
      }
      const bool q_ok = mbar_wait_b(qbar, 0, a.err, sAbort, a.wait_ns);
      if (q_ok && n_it > 0) {
        const uint32_t idesc = F8Q ? idesc_e4m3(kTile, N) : idesc_bf16(kTile, N, false, false);
        const uint32_t bBase = smem_u32(sB);
        bool s_ok = true;
        if constexpr (MX) {  // the query side's scales, stored by the first epilogue group
          s_ok = mbar_wait_b(sbar, 0, a.err, sAbort, a.wait_ns);
          tc_fence_after();
        }
        int committed = 0;
        for (int it = 0; s_ok && it < n_it; ++it) {
          const int st = it % S, acc = it % NA;
          if (!mbar_wait_b(&full[st], (it / S) & 1, a.err, sAbort, a.wait_ns)) break;
          if (!mbar_wait_b(&tempty[acc], ((it / NA) & 1) ^ 1, a.err, sAbort, a.wait_ns)) break;
          tc_fence_after();
          const uint32_t aBase = smem_u32(sA + static_cast<size_t>(st) * L.stage_bytes);
          const uint32_t d = tmem + static_cast<uint32_t>(acc * N);
          if constexpr (MX) {
            // the tile's key scales into this accumulator's group, then D = k . hi (+)= k . lo
            // with the key scale byte of K block ks & 3
            const uint32_t sfa = tmem + sf0 + 8u * static_cast<uint32_t>(acc);
            tmem_cp_32x128b_w4(sfa, smem_desc_plain(smem_u32(sSc + static_cast<size_t>(st) * kMxScaleSlot)));
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t koff = (ks & 3) * 32u;
              const uint32_t boff = (ks >> 2) * static_cast<uint32_t>(N * 128) + koff;
              mma_mx(d, smem_desc(aBase + koff, 16, 1024), smem_desc(bBase + boff, 16, 1024),
                     idesc_mx_e2m1_e4m3(kTile, N, static_cast<uint32_t>(ks & 3), 0u), sfa, tmem + sfb_col, ks > 0);
            }
          } else if constexpr (FP8) {
            // D = k . hi (+)= k . lo: the same key descriptors against both query terms
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t koff = (ks & 3) * 32u;
              const uint32_t boff = (ks >> 2) * static_cast<uint32_t>(N * 128) + koff;
              mma_f8(d, smem_desc(aBase + koff, 16, 1024), smem_desc(bBase + boff, 16, 1024), idesc, ks > 0);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t off = (ks >> 2) * 16384u + (ks & 3) * 32u;
              const uint32_t boff = (ks >> 2) * static_cast<uint32_t>(N * 128) + (ks & 3) * 32u;
              mma_bf16(d, smem_desc(aBase + off, 16, 1024), smem_desc(bBase + boff, 16, 1024), idesc, ks > 0);
            }
          }
          mma_commit(&empty[st]);
          mma_commit(&tfull[acc]);
          ++committed;
        }
        if (committed > 0) wait_time_only(&tfull[(committed - 1) % NA], ((committed - 1) / NA) & 1);
      }
      if (!q_ok && !img_cta) wait_time_only(qbar, 0);  // the image copy must land before the CTA exits
    }
  } else {
    // ---- epilogue: group gp (0/1) takes tiles gp, gp + 2, ...; warp (warp & 3) owns TMEM
    //      lanes 32q..32q+31, i.e. 32 keys of the tile, and reduces every head of them
    const int q = warp & 3;
    const int gq = (warp - 2) >> 2;
    const int gp = gq & 1, ch = gq >> 1;  // tile parity, query half
    const int gh = (G + 1) / 2;
    const int g_lo = gpt == 2 ? ch * gh : 0, g_hi = gpt == 2 ? min(G, g_lo + gh) : G;
    const int rin = q * 32 + lane;
    uint32_t* hist_row = hist ? a.hist_out + qrow0 * kTopkHistRowWords : nullptr;
    if (MX && gq == 0) {
      // the B scales: 2^0 (byte 127) in 8 columns of this warp's 32 lanes
      const uint32_t sb = tmem + (static_cast<uint32_t>(q * 32) << 16) + sfb_col;
      tmem_st4(sb, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st4(sb + 4u, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(sbar);
    }
    if (img_cta) {
      build_image_cta<F8Q>(a, L, sB, b, tid - 64);
      fence_proxy_async_smem();
      mbar_arrive(qbar);
    }
    if constexpr (FUSE) {
      hist_row = a.fuse.hist + static_cast<size_t>(b) * kTopkHistRowWords;
      // the new key entry, if this CTA scores it (first epilogue group, one channel a thread)
      const bool own_new =
          e_new >= 0 && n_it > 0 && static_cast<int64_t>(tile_lo + (n_it - 1) * tile_step) == e_new / kTile;
      if (own_new && gp == 0) {
        const float sc = decode_new_key<KF>(a, b, e_new, tid - 64, sRed4, 7);
        if (tid == 64) {
          *sNewScale = sc;
          mbar_arrive(kbar);
        }
      }
      // the sequence's new main-KV entry
      if (e_new >= 0) decode_new_kv(a, b, e_new, tid - 64, split, L.n_splits);
    }
    const bool w_ok = __all_sync(0xffffffffu, mbar_wait_b(qbar, 0, a.err, sAbort, a.wait_ns));  // gates landed with the image
    const float* kscale_b = FP8 ? static_cast<const float*>(a.kscale) + static_cast<int64_t>(b) * a.E_cap : nullptr;
    const int32_t* cand_b = !FUSE && a.cand ? a.cand + static_cast<int64_t>(qrow0) * a.n_cand : nullptr;
    // the key row of slot sx: the slot itself, or (candidate mode) its position (-1: none)
    auto pos_of = [&](int64_t sx) -> int64_t {
      if (FUSE || !cand_b) return sx;
      return sx < a.n_cand ? static_cast<int64_t>(cand_b[sx]) : -1;
    };
    auto scale_of = [&](int itx) -> float {
      const int64_t px = pos_of(static_cast<int64_t>(tile_lo + itx * tile_step) * kTile + rin);
      return (FP8 && itx < n_it && (FUSE || px >= 0) && px < a.E_cap) ? kscale_b[px] : 1.f;
    };
    float ks_next = scale_of(gp);  // e4m3 key scales, prefetched one tile of this group ahead
    for (int it = gp; w_ok && ch < gpt && it < n_it; it += 2) {
      const int acc = it % NA;
      const float ksc = ks_next;
      ks_next = scale_of(it + 2);
      // (waits are made warp-uniform: the TMEM loads and the histogram below are warp-wide)
      if (!__all_sync(0xffffffffu, mbar_wait_b(&tfull[acc], (it / NA) & 1, a.err, sAbort, a.wait_ns))) break;
      tc_fence_after();
      // the key in this lane's row: the tile's row rin (MXFP4 tiles hold key 4 * lane + q there)
      const int64_t s = static_cast<int64_t>(tile_lo + it * tile_step) * kTile + (MX ? 4 * lane + q : rin);
      float ksc_use = ksc;
      if (FUSE && FP8 && __any_sync(0xffffffffu, s == e_new)) {  // the key compressed in this launch
        if (!__all_sync(0xffffffffu, mbar_wait_b(kbar, 0, a.err, sAbort, a.wait_ns))) break;
        if (s == e_new) ksc_use = *sNewScale;
      }
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * N);
      float res[kMaxG];
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        res[g] = 0.f;
        if (g < g_lo || g >= g_hi) continue;
        float sum = 0.f;
        for (int hc = 0; hc < HI; hc += 32) {
          float v[32];
          tmem_ld32(lane_base + g * HI + hc, v);
          tmem_wait_ld(v);
          sum += relu_dot32(v, sW + g * HI + hc);
        }
        res[g] = sum;
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (s < n_cols) {
        const int64_t ps = pos_of(s);  // the key's position (= s without candidates)
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
          if (g < g_lo || g >= g_hi || g0 + g >= T) continue;
          const float sc = res[g] * ksc_use;
          store_score(a, (qrow0 + g) * a.ld + s, (FUSE || ps >= 0) && ps < sNv[g] ? sc : -INFINITY);
        }
      }
      if (hist && s < n_cols && s < sNv[0]) atomicAdd(&sHist[f2key(stored_score(a, res[0] * ksc_use)) >> 20], 1u);
    }
    if (hist) {
      named_sync(6, 32 * EPI);
      uint32_t* rh = hist_row;
      // the CTAs of a row start their flush at different bins, so that their atomics meet
      // different addresses at the same time
      const int rot = (split * 256) & (kTopkHistBins - 1);
      for (int j = tid - 64; j < kTopkHistBins; j += 32 * EPI) {
        const int i = (j + rot) & (kTopkHistBins - 1);
        const uint32_t c = sHist[i];
        if (c) atomicAdd(&rh[i], c);
      }
      if (!fuse && tid - 64 < kTopkHistCoarse) {
        const int cb = tid - 64;
        constexpr int per = kTopkHistBins / kTopkHistCoarse;
        uint32_t c = 0;
        for (int j = 0; j < per; ++j) c += sHist[cb * per + j];
        if (c) atomicAdd(&rh[kTopkHistBins + cb], c);
      }
    }
  }

  pdl_trigger();  // the next kernel may start launching while this CTA tears down
  // decode step: completing only after the previous kernel keeps the stream order transitive
  if (fuse) pdl_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L.tmem_cols);
  }
}

TcLayout plan_tc(const IndexerArgs& a) {
  TcLayout L{};
  const bool fp8 = a.kidx == CSA_E4M3;
  const bool mx = a.kidx == CSA_MXFP4;
  L.G = std::max(1, std::min({256 / a.HI, a.T, kMaxG}));
  // MXFP4 keys also keep scale groups in TMEM (8 columns per accumulator + 8): two
  // accumulators and those must fit the CTA's share
  if (mx) L.G = std::max(1, std::min(L.G, (512 - 24) / (2 * a.HI)));
  const int64_t n_cols = a.cand ? a.n_cand : a.E_cap;  // candidate slots or cache positions
  const int tiles = static_cast<int>((n_cols + kTile - 1) / kTile);
  auto groups_of = [&](int G) { return static_cast<int64_t>(a.B) * ((a.T + G - 1) / G); };
  // few long rows (decode): two CTAs per SM, key range split over them
  bool decode_like = groups_of(L.G) < a.num_sms;
  if (mx && decode_like) {
    L.G = std::max(1, std::min(L.G, (256 - 24) / (2 * a.HI)));
    decode_like = groups_of(L.G) < a.num_sms;
  }
  L.N = L.G * a.HI;
  L.b_bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(L.N) * 256, 1024));  // bf16 rows or hi+lo
  L.w_bytes = static_cast<uint32_t>(align_up(static_cast<size_t>(L.N) * 4, 16));
  L.stage_bytes = (fp8 || mx) ? kKeyTileBytesF8 : 32768u;
  L.n_qgroups = (a.T + L.G - 1) / L.G;
  const int64_t groups = groups_of(L.G);
  const size_t misc = 1024 + align_up(L.w_bytes, 1024) + 64 + 32 * 8 + 64 +
                      ((a.hist_out || a.fuse.on) && L.G == 1 ? kTopkHistBins * 4 : 0);
  const size_t budget = decode_like ? (113 * 1024) : (227 * 1024);
  const size_t per_stage = L.stage_bytes + (mx ? kMxScaleSlot : 0);
  int S = static_cast<int>((budget - misc - L.b_bytes) / per_stage);
  S = std::max(2, std::min(S, 8));
  L.stages = S;
  L.wide = !decode_like;  // one CTA per SM
  L.smem_bytes = static_cast<uint32_t>(misc + L.b_bytes + static_cast<size_t>(S) * per_stage);
  // as many accumulators (2..4) as the TMEM share of this CTA (512 columns per SM) holds
  const int share = decode_like ? 256 : 512;
  auto cols_needed = [&](int na) {
    const int acc = na * L.N;
    return mx ? ((acc + 7) & ~7) + 8 * na + 8 : acc;
  };
  L.n_acc = 2;
  while (L.n_acc < 4 && cols_needed(L.n_acc + 1) <= share) ++L.n_acc;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(cols_needed(L.n_acc))) cols <<= 1;
  L.tmem_cols = cols;
  if (decode_like) {
    const int64_t target = 2 * static_cast<int64_t>(a.num_sms);
    L.n_splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(target / groups, tiles)));
  } else {
    L.n_splits = 1;
  }
  return L;
}

}  // namespace

IndexerLayout indexer_layout(const IndexerArgs& a) { return plan_tc(a); }


bool indexer_uses_tensor_cores(const IndexerArgs& a) {
  if (a.act != CSA_BF16 || a.dI != 128) return false;
  // MXFP4 keys: dense key ranges, 32 or 64 heads (the TMEM scale groups need the room)
  if (a.kidx == CSA_MXFP4) return a.cand == nullptr && (a.HI == 32 || a.HI == 64);
  // candidate lists on the tensor cores for one query per sequence (the CSA2 Reindex step)
  return (a.cand == nullptr || (a.T == 1 && !a.fuse.on && a.hist_out == nullptr)) &&
         (a.HI == 32 || a.HI == 64 || a.HI == 128) && (a.kidx == CSA_BF16 || a.kidx == CSA_E4M3);
}

size_t indexer_workspace_bytes(const IndexerArgs& a) {
  if (!indexer_uses_tensor_cores(a) || a.B * a.T == 0) return 0;
  const TcLayout L = plan_tc(a);
  return static_cast<size_t>(a.B) * L.n_qgroups * (L.b_bytes + L.w_bytes);
}

cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T;
  const int64_t n_cols = a.cand ? a.n_cand : a.E_cap;
  if (rows == 0 || n_cols == 0) return cudaSuccess;
  if (indexer_uses_tensor_cores(a)) {
    const int kf = a.kidx == CSA_MXFP4 ? kKeyMx : a.kidx == CSA_E4M3 ? kKeyE4m3 : kKeyBf16;
    const bool f8q = kf != kKeyBf16;
    const TcLayout L = plan_tc(a);
    CUtensorMap map;
    bool enc;
    if (kf == kKeyMx) {
      // packed E2M1 payload (64 B a key) unpacked by TMA into 8-bit slots; a 3D view whose box
      // (128 codes, 1, 32) at (0, c, r) takes keys 4(r + l) + c, l = 0..31
      const uint64_t dims[3] = {128, 4, static_cast<uint64_t>(a.B) * a.E_cap / 4};
      const uint64_t strides[2] = {64, 256};
      const uint32_t box[3] = {128, 1, 32};
      enc = encode_tmap_generic(&map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(a.kI), dims, strides,
                                box, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      enc = encode_tmap_2d(&map, kf == kKeyE4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           const_cast<void*>(a.kI), 128, static_cast<uint64_t>(a.B) * a.E_cap, kf == kKeyE4m3 ? 128 : 256,
                           kf == kKeyE4m3 ? 128 : 64, kTile);
    }
    if (!enc) return cudaErrorInvalidValue;
    uint8_t* images = static_cast<uint8_t*>(a.ws);
    cudaError_t e = cudaSuccess;
    if (!a.images_ready && !image_in_cta(a, L)) {
      dim3 gq(L.n_qgroups, a.B, (L.N + 7) / 8);
      e = f8q ? launch_pdl(indexer_qprep_kernel<true>, gq, dim3(256), 0, s, a, L, images)
              : launch_pdl(indexer_qprep_kernel<false>, gq, dim3(256), 0, s, a, L, images);
      count_launches(1);
      if (e != cudaSuccess) return e;
    }
    dim3 grid(L.n_splits, L.n_qgroups, a.B);
    static std::atomic<unsigned long long> attr{0};
    if (first_use_in_context(attr)) {
      const int mx = 227 * 1024;
#define CSA_IDX_ATTR(KF, FU, MB) \
  cudaFuncSetAttribute(indexer_tc_kernel<KF, FU, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)
      CSA_IDX_ATTR(kKeyBf16, false, 2); CSA_IDX_ATTR(kKeyE4m3, false, 2); CSA_IDX_ATTR(kKeyMx, false, 2);
      CSA_IDX_ATTR(kKeyBf16, true, 2);  CSA_IDX_ATTR(kKeyE4m3, true, 2);  CSA_IDX_ATTR(kKeyMx, true, 2);
      CSA_IDX_ATTR(kKeyBf16, false, 1); CSA_IDX_ATTR(kKeyE4m3, false, 1); CSA_IDX_ATTR(kKeyMx, false, 1);
#undef CSA_IDX_ATTR
    }
    const uint8_t* cimages = images;
    const dim3 blk(L.wide && !a.fuse.on ? tc_threads(1) : tc_threads(2));
    const size_t sm = L.smem_bytes;
#define CSA_IDX_LAUNCH(FU, MB)                                                                               \
  (kf == kKeyMx     ? launch_pdl(indexer_tc_kernel<kKeyMx, FU, MB>, grid, blk, sm, s, map, a, L, cimages, n_cols)   \
   : kf == kKeyE4m3 ? launch_pdl(indexer_tc_kernel<kKeyE4m3, FU, MB>, grid, blk, sm, s, map, a, L, cimages, n_cols) \
                    : launch_pdl(indexer_tc_kernel<kKeyBf16, FU, MB>, grid, blk, sm, s, map, a, L, cimages, n_cols))
    if (a.fuse.on)
      e = CSA_IDX_LAUNCH(true, 2);
    else if (L.wide)
      e = CSA_IDX_LAUNCH(false, 1);
    else
      e = CSA_IDX_LAUNCH(false, 2);
#undef CSA_IDX_LAUNCH
    count_launches(1);
    return e;
  }
  dim3 grid(static_cast<unsigned>((n_cols + 127) / 128), static_cast<unsigned>(rows));
  const size_t smem = static_cast<size_t>(a.HI) * (a.dI + 1) * 4;
#define CSA_SIMT(TQ, TK, DI)                                                                          \
  do {                                                                                                \
    cudaFuncSetAttribute(indexer_simt_kernel<TQ, TK, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                         static_cast<int>(smem));                                                     \
    indexer_simt_kernel<TQ, TK, DI><<<grid, 128, smem, s>>>(a, n_cols);                              \
  } while (0)
#define CSA_SIMT_DI(TQ, TK)         \
  do {                              \
    if (a.dI == 32)                 \
      CSA_SIMT(TQ, TK, 32);         \
    else if (a.dI == 64)            \
      CSA_SIMT(TQ, TK, 64);         \
    else                            \
      CSA_SIMT(TQ, TK, 128);        \
  } while (0)
  if (a.kidx == CSA_MXFP4) {  // bf16 queries, dI = 128 (checked by the caller)
    CSA_SIMT(__nv_bfloat16, MxKey, 128);
  } else if (a.act == CSA_F32) {
    if (a.kidx == CSA_E4M3)
      CSA_SIMT_DI(float, uint8_t);
    else
      CSA_SIMT_DI(float, float);
  } else {
    if (a.kidx == CSA_E4M3)
      CSA_SIMT_DI(__nv_bfloat16, uint8_t);
    else
      CSA_SIMT_DI(__nv_bfloat16, __nv_bfloat16);
  }
#undef CSA_SIMT_DI
#undef CSA_SIMT
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace csa
