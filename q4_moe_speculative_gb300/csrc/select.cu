// select.cu — compressed-attention block selection: compaction of the admitted index
// (K6), scoring of admitted blocks only (K5) and the bounded radix top-k (K7).
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)",
// paragraph "Decode at depth": compressed attention picks 512 blocks per layer; layers
// score only the blocks their mask admits, compact the admitted index once per row and
// select the top 512 with a bounded radix select.
//
// Order of the chain on the device: K6 (per-row admitted counts, exclusive offsets per
// mask word, admitted index) -> K5 (scores, written at the compacted position) -> K7.
//
// Two scoring modes give the same selection:
//  * canonical: K5 computes every admitted block's score in the canonical fp32 order
//    (fmaf over i ascending, then over heads ascending) on CUDA cores; K7 radix-selects.
//  * tensor-core (default): K5 computes q_h . k for all rows and heads of a 128-block tile
//    as one [128 x 128] x [128 x R*Hh] bf16 contraction on tcgen05 (TMA-staged operands,
//    fp32 accumulators in TMEM) and writes, per admitted block, a certified interval
//    [lo, hi] that contains the canonical score: |s_tc - s_canon| <= eps with
//    eps = 2^-10 * ||k|| * sum_h |w_h| ||q_h||  (the two dot products differ by at most a
//    few hundred fp32 roundings of terms bounded by |q_i k_i|, and the canonical sum of
//    |q_i k_i| is at most ||q|| ||k||; 2^-10 leaves a margin of about 2^7 over that).
//    K7 takes T = k-th largest lo; every block of the canonical top-k has hi >= T, so it
//    re-scores only the candidates with hi >= T in the canonical order and selects among
//    them exactly. The result is identical to the canonical mode by construction.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace dsmoe {
namespace {

constexpr int kCompactThreads = 1024;
constexpr int kScoreThreads = 128;   // one key per thread, one tile of keys per CTA
constexpr int kScoreMaxHeads = 16;
constexpr int kTopkThreads = 1024;
constexpr int kResidCap = 4096;      // residual radix bucket kept in shared memory
constexpr int kCandCap = 4096;       // re-score candidates kept in shared memory
constexpr uint32_t kWaitPolls = 1u << 17;   // bounded mbarrier polling (<= ~0.13 s)
constexpr float kEpsRel = 0.0009765625f;    // 2^-10

// Exclusive block-wide prefix sum of v over blockDim.x (<= 1024) threads; *total gets
// the sum. Uses `scratch` (>= 33 ints of shared memory). All threads must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    scratch[lane] = wi - w;          // exclusive prefix of warp totals
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  const int res = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// Admitted bits of mask word wi for a row with limit lim (bits at b >= lim cleared).
__device__ __forceinline__ uint32_t admitted_word(const uint32_t* m, int wi, int lim) {
  const int b0 = wi * 32;
  if (b0 >= lim) return 0u;
  uint32_t w = m[wi];
  const int rem = lim - b0;
  if (rem < 32) w &= (1u << rem) - 1u;
  return w;
}

// Order-preserving 32-bit key of an fp32 score: larger score -> larger key, -0 == +0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Canonical score of one block: q [Hh][128] fp32 (shared), key 128 bf16 (global), w [Hh].
__device__ __forceinline__ float canonical_score(const float* q, const uint16_t* key,
                                                 const float* w, int Hh) {
  float d[kScoreMaxHeads];
#pragma unroll
  for (int h = 0; h < kScoreMaxHeads; ++h) d[h] = 0.0f;
  const uint4* k4 = reinterpret_cast<const uint4*>(key);
  for (int c = 0; c < 16; ++c) {
    const uint4 kv = __ldg(k4 + c);
    const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                         bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
    for (int h = 0; h < kScoreMaxHeads; ++h) {
      if (h < Hh) {
        const float* qh = q + h * 128 + c * 8;
        float t = d[h];
#pragma unroll
        for (int e = 0; e < 8; ++e) t = __fmaf_rn(qh[e], kf[e], t);
        d[h] = t;
      }
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < kScoreMaxHeads; ++h)
    if (h < Hh) s = __fmaf_rn(w[h], d[h] > 0.0f ? d[h] : 0.0f, s);
  return s;
}

// ---------------------------------------------------------------------------------
// K6: compaction once per (layer, row). One CTA per row: popcount + block scan of the
// admitted words gives every word's exclusive offset (kept for K5) and the count; each
// warp then scatters the admitted indices of 32 words with a ballot over per-lane
// predicates (bit set and block below the causal limit).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kCompactThreads)
    k6_compact(int R, int N, const uint32_t* __restrict__ mask, const int32_t* __restrict__ limit,
               int32_t* __restrict__ wordoff, int32_t* __restrict__ cidx,
               int32_t* __restrict__ ccount) {
  __shared__ int scratch[33];
  __shared__ int s_off[kCompactThreads];
  const int lr = blockIdx.x;
  const int W = (N + 31) >> 5;
  const uint32_t* m = mask + (size_t)lr * W;
  int lim = limit[lr];
  lim = lim < 0 ? 0 : (lim > N ? N : lim);
  int32_t* wo = wordoff + (size_t)lr * W;
  int32_t* ci = cidx + (size_t)lr * N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int base = 0;
  for (int c0 = 0; c0 < W; c0 += kCompactThreads) {
    const int wi = c0 + tid;
    const uint32_t mw = (wi < W) ? admitted_word(m, wi, lim) : 0u;
    int total;
    const int excl = base + block_excl_scan(__popc(mw), scratch, &total);
    if (wi < W) wo[wi] = excl;
    s_off[tid] = excl;
    __syncthreads();
    for (int q = warp; q < kCompactThreads && c0 + q < W; q += kCompactThreads / 32) {
      const int w = c0 + q;
      const int b = w * 32 + lane;
      const bool pred = (b < lim) && ((m[w] >> lane) & 1u);
      const uint32_t bal = __ballot_sync(0xffffffffu, pred);
      if (pred) ci[s_off[q] + __popc(bal & ((1u << lane) - 1u))] = b;
    }
    base += total;
    __syncthreads();
  }
  if (tid == 0) ccount[lr] = base;
}

struct ScoreArgs {
  int L, R, Hh, N;
  int64_t key_stride;
  const uint16_t* keys;
  const uint16_t* q;
  const float* hw;
  const uint32_t* mask;
  const int32_t* limit;
  const int32_t* wordoff;
  uint32_t* sc0;      // canonical: fp32 scores; tensor-core: keys of the lower bounds
  float* sc1;         // tensor-core: upper bounds
  uint32_t* status;
};

// Rows (bit r) of the layer that admit block b.
__device__ __forceinline__ uint32_t admitting_rows(const ScoreArgs& a, int l, int b, int W) {
  uint32_t rows = 0;
  if (b < a.N) {
    for (int r = 0; r < a.R; ++r) {
      const size_t lr = (size_t)l * a.R + r;
      const int lim = a.limit[lr];
      if (b < lim && ((a.mask[lr * W + (b >> 5)] >> (b & 31)) & 1u)) rows |= 1u << r;
    }
  }
  return rows;
}

__device__ __forceinline__ int compact_pos(const ScoreArgs& a, size_t lr, int b, int W) {
  const int wi = b >> 5;
  const uint32_t mw = admitted_word(a.mask + lr * W, wi, a.limit[lr]);
  return a.wordoff[lr * W + wi] + __popc(mw & ((1u << (b & 31)) - 1u));
}

// ---------------------------------------------------------------------------------
// K5 (canonical mode): CUDA-core scoring of admitted blocks. CTA = (layer, 128 blocks);
// a key is loaded only if some row admits it, once for all rows.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kScoreThreads) k5_score(ScoreArgs a) {
  extern __shared__ float smem[];
  const int R = a.R, Hh = a.Hh, D = 128;
  float* qs = smem;                                        // [R][Hh][D]
  float* ws = qs + R * Hh * D;                             // [R][Hh]
  uint4* ks = reinterpret_cast<uint4*>(ws + ((R * Hh + 3) & ~3));  // [128 keys][16 chunks]
  __shared__ uint32_t s_rows[kScoreThreads];

  const int tiles = (a.N + kScoreThreads - 1) / kScoreThreads;
  const int l = blockIdx.x / tiles;
  const int tile = blockIdx.x - l * tiles;
  const int tid = threadIdx.x;
  const int b = tile * kScoreThreads + tid;
  const int W = (a.N + 31) >> 5;

  const uint32_t rows = admitting_rows(a, l, b, W);
  s_rows[tid] = rows;
  const int any = __syncthreads_or(rows != 0);
  if (!any) return;

  for (int i = tid; i < R * Hh * D / 2; i += blockDim.x) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(a.q + (size_t)l * R * Hh * D)[i];
    qs[2 * i] = bf16_lo(w);
    qs[2 * i + 1] = bf16_hi(w);
  }
  for (int i = tid; i < R * Hh; i += blockDim.x) ws[i] = a.hw[(size_t)l * R * Hh + i];
  const uint16_t* kbase = a.keys + (size_t)l * a.key_stride;
  for (int i = tid; i < kScoreThreads * 16; i += blockDim.x) {
    const int kk = i >> 4, c = i & 15;
    const int bb = tile * kScoreThreads + kk;
    if (s_rows[kk] != 0u)
      ks[kk * 16 + (c ^ (kk & 15))] = ldg_stream(kbase + (size_t)bb * D + c * 8);
  }
  __syncthreads();
  if (rows == 0u) return;

  for (int r = 0; r < R; ++r) {
    if (!(rows & (1u << r))) continue;
    float d[kScoreMaxHeads];
#pragma unroll
    for (int h = 0; h < kScoreMaxHeads; ++h) d[h] = 0.0f;
    const float* qr = qs + r * Hh * D;
    for (int c = 0; c < 16; ++c) {
      const uint4 kv = ks[tid * 16 + (c ^ (tid & 15))];
      const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                           bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
      for (int h = 0; h < kScoreMaxHeads; ++h) {
        if (h < Hh) {
          const float4 q0 = *reinterpret_cast<const float4*>(qr + h * D + c * 8);
          const float4 q1 = *reinterpret_cast<const float4*>(qr + h * D + c * 8 + 4);
          float t = d[h];
          t = __fmaf_rn(q0.x, kf[0], t); t = __fmaf_rn(q0.y, kf[1], t);
          t = __fmaf_rn(q0.z, kf[2], t); t = __fmaf_rn(q0.w, kf[3], t);
          t = __fmaf_rn(q1.x, kf[4], t); t = __fmaf_rn(q1.y, kf[5], t);
          t = __fmaf_rn(q1.z, kf[6], t); t = __fmaf_rn(q1.w, kf[7], t);
          d[h] = t;
        }
      }
    }
    float s = 0.0f;
#pragma unroll
    for (int h = 0; h < kScoreMaxHeads; ++h)
      if (h < Hh) s = __fmaf_rn(ws[r * Hh + h], d[h] > 0.0f ? d[h] : 0.0f, s);
    const size_t lr = (size_t)l * R + r;
    reinterpret_cast<float*>(a.sc0)[lr * (size_t)a.N + compact_pos(a, lr, b, W)] = s;
  }
}

// ---------------------------------------------------------------------------------
// K5 (tensor-core mode): CTA = (layer, 128 blocks), 4 warps. TMA brings the 128 keys
// [128 x 128 bf16] and the layer's queries [R*Hh (padded to NCH*16) x 128 bf16] into
// shared memory in the 128-byte swizzled K-major layout; one thread issues 8 tcgen05.mma
// (M = 128 keys, N = R*Hh, K = 16 each) into a TMEM accumulator; each warp reads its 32
// lanes (one key per thread) and forms the approximate score and its certified interval.
// Every wait is bounded; on give-up the kernel flags a timeout, waits once more (bounded)
// for its own copies / MMAs, frees TMEM and returns.
// ---------------------------------------------------------------------------------
template <int NCH>
__global__ void __launch_bounds__(kScoreThreads)
    k5_score_tc(const __grid_constant__ CUtensorMap tm_keys,
                const __grid_constant__ CUtensorMap tm_q, ScoreArgs a) {
  constexpr int NPAD = NCH * 16;
  constexpr uint32_t kTmemCols = NPAD <= 32 ? 32 : (NPAD <= 64 ? 64 : 128);
  constexpr uint32_t kKeyBytes = 128 * 128 * 2;
  constexpr uint32_t kQChunk = NPAD * 128;          // one 64-column half of the queries
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_tma, bar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ uint32_t s_rows[kScoreThreads];
  __shared__ float s_qn[NPAD];
  __shared__ float s_w[NPAD];
  __shared__ float s_F[8];

  const int R = a.R, Hh = a.Hh, RH = R * Hh;
  const int tiles = (a.N + kScoreThreads - 1) / kScoreThreads;
  const int l = blockIdx.x / tiles;
  const int tile = blockIdx.x - l * tiles;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = tile * kScoreThreads + tid;
  const int W = (a.N + 31) >> 5;

  const uint32_t rows = admitting_rows(a, l, b, W);
  s_rows[tid] = rows;
  const int any = __syncthreads_or(rows != 0);
  if (!any) return;

  // 1024-byte aligned operand tiles inside the dynamic shared memory.
  const uint32_t raw = sm100::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* tile_keys = smem_raw + (base - raw);
  uint8_t* tile_q = tile_keys + kKeyBytes;

  if (tid == 0) {
    sm100::prefetch_tensormap(&tm_keys);
    sm100::prefetch_tensormap(&tm_q);
    sm100::mbar_init(&bar_tma, 1);
    sm100::mbar_init(&bar_mma, 1);
    sm100::fence_mbar_init();
  }
  if (warp == 0) {
    sm100::tmem_alloc(&s_tmem, kTmemCols);
    sm100::tmem_relinquish();
  }
  if (tid < NPAD) s_w[tid] = tid < RH ? a.hw[(size_t)l * RH + tid] : 0.0f;
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (tid == 0) {
    sm100::mbar_arrive_expect_tx(&bar_tma, kKeyBytes + 2 * kQChunk);
    sm100::tma_load_3d(tile_keys, &tm_keys, 0, tile * 128, l, &bar_tma);
    sm100::tma_load_3d(tile_keys + kKeyBytes / 2, &tm_keys, 64, tile * 128, l, &bar_tma);
    sm100::tma_load_2d(tile_q, &tm_q, 0, l * RH, &bar_tma);
    sm100::tma_load_2d(tile_q + kQChunk, &tm_q, 64, l * RH, &bar_tma);
  }
  bool ok = sm100::mbar_wait(&bar_tma, 0, kWaitPolls);
  if (!ok) {
    if (tid == 0) flag_status(a.status, kStatusTimeout);
    sm100::mbar_wait(&bar_tma, 0, kWaitPolls);    // let our own copies land before exit
  }
  if (ok && tid == 0) {
    constexpr uint32_t idesc = sm100::idesc_bf16_f32(128, NPAD);
    const uint32_t ka = sm100::smem_u32(tile_keys), qa = sm100::smem_u32(tile_q);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t half = (uint32_t)(kk >> 2), step = (uint32_t)(kk & 3) * 32u;
      const uint64_t ad = sm100::desc_k_sw128(ka + half * (kKeyBytes / 2) + step);
      const uint64_t bd = sm100::desc_k_sw128(qa + half * kQChunk + step);
      sm100::mma_bf16(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
    sm100::mma_commit(&bar_mma);
  }
  if (ok) {
    ok = sm100::mbar_wait(&bar_mma, 0, kWaitPolls);
    if (!ok) {
      if (tid == 0) flag_status(a.status, kStatusTimeout);
      sm100::mbar_wait(&bar_mma, 0, kWaitPolls);
    }
  }
  sm100::tc_fence_after();

  if (ok) {
    // Query norms (upper bounds) and the per-row factor F_r = sum_h |w_h| ||q_h||.
    if (tid < NPAD) {
      float ss = 0.0f;
      const uint4* row0 = reinterpret_cast<const uint4*>(tile_q + tid * 128);
      const uint4* row1 = reinterpret_cast<const uint4*>(tile_q + kQChunk + tid * 128);
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint4 u0 = row0[g], u1 = row1[g];
        const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float lo = bf16_lo(wv[e]), hi = bf16_hi(wv[e]);
          ss = __fmaf_ru(lo, lo, ss);
          ss = __fmaf_ru(hi, hi, ss);
        }
      }
      s_qn[tid] = __fmul_ru(__fsqrt_ru(ss), 1.0000153f);   // (1 + 2^-16) margin
    }
    __syncthreads();
    if (tid < R) {
      float F = 0.0f;
      for (int h = 0; h < Hh; ++h) F = __fmaf_ru(fabsf(s_w[tid * Hh + h]), s_qn[tid * Hh + h], F);
      s_F[tid] = F;
    }
    __syncthreads();

    // This thread's key norm (order of the 16-byte granules does not matter).
    float kss = 0.0f;
    {
      const uint8_t* kr0 = tile_keys + tid * 128;
      const uint8_t* kr1 = tile_keys + kKeyBytes / 2 + tid * 128;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const int gg = (g + tid) & 7;   // rotate to spread the banks
        const uint4 u0 = *reinterpret_cast<const uint4*>(kr0 + gg * 16);
        const uint4 u1 = *reinterpret_cast<const uint4*>(kr1 + gg * 16);
        const uint32_t wv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float lo = bf16_lo(wv[e]), hi = bf16_hi(wv[e]);
          kss = __fmaf_ru(lo, lo, kss);
          kss = __fmaf_ru(hi, hi, kss);
        }
      }
    }
    const float kn = __fmul_ru(__fsqrt_ru(kss), 1.0000153f);

    float d[NPAD];
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int c = 0; c < NCH; ++c) sm100::tmem_ld16(lane_base + (uint32_t)(c * 16), d + c * 16);

    if (rows != 0u) {
      float s = 0.0f;
      int r = 0, h = 0;
#pragma unroll
      for (int p = 0; p < NPAD; ++p) {
        if (p < RH) {
          if (h == 0) s = 0.0f;
          s = __fmaf_rn(s_w[p], d[p] > 0.0f ? d[p] : 0.0f, s);
          if (h == Hh - 1) {
            if (rows & (1u << r)) {
              const size_t lr = (size_t)l * R + r;
              const float eps = __fmul_ru(__fmul_ru(kEpsRel, kn), s_F[r]);
              const int pos = compact_pos(a, lr, b, W);
              a.sc0[lr * (size_t)a.N + pos] = score_key(__fsub_rd(s, eps));
              a.sc1[lr * (size_t)a.N + pos] = __fadd_ru(s, eps);
            }
            h = 0;
            ++r;
          } else {
            ++h;
          }
        }
      }
    }
  }
  (void)lane;
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------
// Radix threshold: the key of the need-th largest element among n keys, found MSB-first
// 8 bits at a time. `key_at(i)` gives the key of element i. After the first two passes the
// elements whose top 16 bits match are gathered into `r_key` (if at most kResidCap of
// them) and the last two passes run there. On return *need_out = how many elements equal
// to the threshold belong to the selection. All threads must call it.
// ---------------------------------------------------------------------------------
template <typename KeyAt>
__device__ uint32_t radix_threshold(int n, int need, KeyAt key_at, int* hist, int* scratch,
                                    uint32_t* r_key, int* s_misc, uint32_t* status,
                                    int* need_out) {
  const int tid = threadIdx.x;
  int& s_bucket = s_misc[0];
  int& s_need = s_misc[1];
  int& s_rn = s_misc[2];
  uint32_t prefix = 0;
  bool resid = false;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    if (tid == 0) {
      s_bucket = -1;
      s_need = need;
    }
    __syncthreads();
    if (resid) {
      const int rn = s_rn < kResidCap ? s_rn : kResidCap;
      for (int i = tid; i < rn; i += blockDim.x) {
        const uint32_t key = r_key[i];
        if ((key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
    } else {
      for (int i = tid; i < n; i += blockDim.x) {
        const uint32_t key = key_at(i);
        if (pass == 0 || (key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
    }
    __syncthreads();
    {
      const int v = tid < 256 ? hist[255 - tid] : 0;
      int total;
      const int excl = block_excl_scan(v, scratch, &total);
      if (tid < 256 && excl < need && need <= excl + v) {
        s_bucket = 255 - tid;
        s_need = need - excl;
      }
    }
    __syncthreads();
    if (s_bucket < 0) {  // histogram inconsistent with `need`: report, keep indices valid
      if (tid == 0) {
        flag_status(status, kStatusCheck);
        s_bucket = 0;
      }
      __syncthreads();
    }
    prefix = (prefix << 8) | (uint32_t)s_bucket;
    need = s_need;
    if (pass == 1 && !resid) {
      const int cnt = hist[s_bucket];
      if (cnt <= kResidCap) {
        if (tid == 0) s_rn = 0;
        __syncthreads();
        for (int i = tid; i < n; i += blockDim.x) {
          const uint32_t key = key_at(i);
          if ((key >> 16) == prefix) {
            const int p = atomicAdd(&s_rn, 1);
            if (p < kResidCap) r_key[p] = key;
          }
        }
        __syncthreads();
        resid = true;
        if (s_rn != cnt && tid == 0) flag_status(status, kStatusCheck);
      }
    }
    __syncthreads();
  }
  *need_out = need;
  return prefix;
}

// Writes, in array order, every element with key > T and the first `need` elements with
// key == T: out[j] = idx_at(i). Returns the number written (<= K).
template <typename KeyAt, typename IdxAt>
__device__ int ordered_take(int n, int K, uint32_t T, int need, KeyAt key_at, IdxAt idx_at,
                            int32_t* out, int* scratch) {
  int taken = 0, eq_seen = 0;
  for (int c0 = 0; c0 < n && taken < K; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    uint32_t key = 0;
    if (i < n) key = key_at(i);
    const int gt = (i < n) && key > T;
    const int eq = (i < n) && key == T;
    int eq_total;
    const int eq_rank = eq_seen + block_excl_scan(eq, scratch, &eq_total);
    const int take = gt || (eq && eq_rank < need);
    int take_total;
    const int pos = taken + block_excl_scan(take, scratch, &take_total);
    if (take && pos < K) out[pos] = idx_at(i);
    taken += take_total;
    eq_seen += eq_total;
  }
  return taken;
}

// ---------------------------------------------------------------------------------
// K7: bounded radix top-k per (layer, row), one CTA of 1024 threads.
// Canonical mode: threshold and ordered take over the canonical scores.
// Tensor-core mode: threshold T over the lower bounds; ordered gather of the candidates
// with upper bound >= T (bounded by kCandCap); canonical re-score of the candidates;
// threshold and ordered take among them. Above the bound: canonical re-score of every
// admitted block of the row, then the canonical-mode path.
// ---------------------------------------------------------------------------------
struct TopkArgs {
  int R, Hh, N, K;
  int64_t key_stride;
  const uint16_t* keys;
  const uint16_t* q;
  const float* hw;
  const int32_t* cidx;
  const int32_t* ccount;
  uint32_t* sc0;
  const float* sc1;
  int32_t* sel;
  int32_t* nsel;
  uint32_t* status;
  int tc_mode;
};

__global__ void __launch_bounds__(kTopkThreads) k7_topk(TopkArgs a) {
  __shared__ int hist[256];
  __shared__ int scratch[33];
  __shared__ int s_misc[4];
  __shared__ uint32_t r_key[kResidCap];
  extern __shared__ uint8_t dsm[];
  int32_t* cand = reinterpret_cast<int32_t*>(dsm);               // [kCandCap] positions
  uint32_t* ckey = reinterpret_cast<uint32_t*>(cand + kCandCap);  // [kCandCap] keys
  float* qf = reinterpret_cast<float*>(ckey + kCandCap);          // [Hh][128]
  float* wf = qf + kScoreMaxHeads * 128;                          // [Hh]

  const int lr = blockIdx.x;
  const int l = lr / a.R;
  const int tid = threadIdx.x;
  const int n = a.ccount[lr];
  const int K = a.K;
  const int32_t* ci = a.cidx + (size_t)lr * a.N;
  uint32_t* s0 = a.sc0 + (size_t)lr * a.N;
  int32_t* out = a.sel + (size_t)lr * K;

  if (n <= K) {
    for (int i = tid; i < K; i += blockDim.x) out[i] = i < n ? ci[i] : -1;
    if (tid == 0) a.nsel[lr] = n;
    return;
  }

  auto idx_at = [&](int i) { return ci[i]; };
  const uint16_t* kbase = a.keys + (size_t)l * a.key_stride;
  bool canonical = !a.tc_mode;

  if (a.tc_mode) {
    const float* s1 = a.sc1 + (size_t)lr * a.N;
    int need;
    const uint32_t T = radix_threshold(
        n, K, [&](int i) { return s0[i]; }, hist, scratch, r_key, s_misc, a.status, &need);
    // Ordered gather of candidates (upper bound can reach T), bounded by kCandCap.
    int m = 0;
    for (int c0 = 0; c0 < n; c0 += blockDim.x) {
      const int i = c0 + tid;
      const int c = (i < n) && score_key(s1[i]) >= T;
      int tot;
      const int p = m + block_excl_scan(c, scratch, &tot);
      if (c && p < kCandCap) cand[p] = i;
      m += tot;
    }
    // Stage this row's queries and weights as fp32.
    const uint16_t* qrow = a.q + (size_t)lr * a.Hh * 128;
    for (int i = tid; i < a.Hh * 128; i += blockDim.x) qf[i] = bf16_bits_to_f32(qrow[i]);
    for (int i = tid; i < a.Hh; i += blockDim.x) wf[i] = a.hw[(size_t)lr * a.Hh + i];
    __syncthreads();
    if (m <= kCandCap) {
      for (int j = tid; j < m; j += blockDim.x) {
        const int b = ci[cand[j]];
        ckey[j] = score_key(canonical_score(qf, kbase + (size_t)b * 128, wf, a.Hh));
      }
      __syncthreads();
      int need2;
      const uint32_t T2 = radix_threshold(
          m, K, [&](int j) { return ckey[j]; }, hist, scratch, r_key, s_misc, a.status, &need2);
      const int taken = ordered_take(
          m, K, T2, need2, [&](int j) { return ckey[j]; }, [&](int j) { return ci[cand[j]]; },
          out, scratch);
      if (tid == 0) {
        a.nsel[lr] = K;
        if (taken != K) flag_status(a.status, kStatusCheck);
      }
      return;
    }
    // Too many candidates (e.g. heavy ties): canonical scores for the whole row.
    for (int i = tid; i < n; i += blockDim.x)
      s0[i] = __float_as_uint(canonical_score(qf, kbase + (size_t)ci[i] * 128, wf, a.Hh));
    __syncthreads();
    canonical = true;
  }

  if (canonical) {
    int need;
    auto key_at = [&](int i) { return score_key(__uint_as_float(s0[i])); };
    const uint32_t T = radix_threshold(n, K, key_at, hist, scratch, r_key, s_misc, a.status, &need);
    const int taken = ordered_take(n, K, T, need, key_at, idx_at, out, scratch);
    if (tid == 0) {
      a.nsel[lr] = K;
      if (taken != K) flag_status(a.status, kStatusCheck);
    }
  }
}

// --------------------------------------------------------------- tensor maps --------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

template <int NCH>
cudaError_t launch_tc(const SelDims& d, const CUtensorMap& tk, const CUtensorMap& tq,
                      const ScoreArgs& a, cudaStream_t s) {
  const size_t smem = 1024 + 128 * 128 * 2 + 2 * (size_t)NCH * 16 * 128;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(k5_score_tc<NCH>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  const int tiles = (d.N + kScoreThreads - 1) / kScoreThreads;
  k5_score_tc<NCH><<<d.L * tiles, kScoreThreads, smem, s>>>(tk, tq, a);
  return cudaGetLastError();
}

}  // namespace

SelLayout sel_layout(const SelDims& d, bool caller_cidx) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t LR = (size_t)d.L * d.R;
  const size_t W = (size_t)(d.N + 31) / 32;
  SelLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  L.wordoff = off; off += up(sizeof(int32_t) * LR * W);
  if (!caller_cidx) {
    L.cidx = off; off += up(sizeof(int32_t) * LR * (size_t)d.N);
    L.ccount = off; off += up(sizeof(int32_t) * LR);
  } else {
    L.cidx = L.ccount = (size_t)-1;
  }
  L.cscore = off; off += up(sizeof(float) * LR * (size_t)d.N);
  L.chi = off; off += up(sizeof(float) * LR * (size_t)d.N);
  L.total = off;
  return L;
}

bool tc_scoring_supported(const SelDims& d, const uint16_t* keys, const uint16_t* q) {
  const int RH = d.R * d.Hh;
  return encode_fn() != nullptr && RH <= 128 && d.D == 128 &&
         (reinterpret_cast<uintptr_t>(keys) % 16) == 0 &&
         (reinterpret_cast<uintptr_t>(q) % 16) == 0 && (d.key_stride % 8) == 0;
}

cudaError_t launch_compact(const SelDims& d, const uint32_t* mask, const int32_t* limit,
                           const SelWorkspace& ws, cudaStream_t s) {
  k6_compact<<<d.L * d.R, kCompactThreads, 0, s>>>(d.R, d.N, mask, limit, ws.wordoff, ws.cidx,
                                                   ws.ccount);
  return cudaGetLastError();
}

cudaError_t launch_score(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                         const float* head_w, const uint32_t* mask, const int32_t* limit,
                         const SelWorkspace& ws, bool tc, cudaStream_t s) {
  ScoreArgs a{d.L, d.R, d.Hh, d.N, d.key_stride, keys, q, head_w, mask, limit, ws.wordoff,
              reinterpret_cast<uint32_t*>(ws.cscore), ws.chi, ws.header};
  if (!tc) {
    const int RH = d.R * d.Hh;
    const size_t smem = sizeof(float) * ((size_t)RH * 128 + ((RH + 3) & ~3)) +
                        (size_t)kScoreThreads * 16 * sizeof(uint4);
    if (smem > 48 * 1024) {
      cudaError_t err = cudaFuncSetAttribute(k5_score, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
      if (err != cudaSuccess) return err;
    }
    const int tiles = (d.N + kScoreThreads - 1) / kScoreThreads;
    k5_score<<<d.L * tiles, kScoreThreads, smem, s>>>(a);
    return cudaGetLastError();
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int RH = d.R * d.Hh;
  const int nch = (RH + 15) / 16;
  CUtensorMap tk, tq;
  {
    const cuuint64_t dims[3] = {128, (cuuint64_t)d.N, (cuuint64_t)d.L};
    const cuuint64_t strides[2] = {256, (cuuint64_t)d.key_stride * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(keys), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {128, (cuuint64_t)d.L * RH};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {64, (cuuint32_t)(nch * 16)};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(q), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  switch (nch) {
    case 1: return launch_tc<1>(d, tk, tq, a, s);
    case 2: return launch_tc<2>(d, tk, tq, a, s);
    case 3: return launch_tc<3>(d, tk, tq, a, s);
    case 4: return launch_tc<4>(d, tk, tq, a, s);
    case 5: return launch_tc<5>(d, tk, tq, a, s);
    case 6: return launch_tc<6>(d, tk, tq, a, s);
    case 7: return launch_tc<7>(d, tk, tq, a, s);
    case 8: return launch_tc<8>(d, tk, tq, a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                        const float* head_w, int32_t* sel, int32_t* nsel,
                        const SelWorkspace& ws, bool tc, cudaStream_t s) {
  TopkArgs a{d.R, d.Hh, d.N, d.topk, d.key_stride, keys, q, head_w, ws.cidx, ws.ccount,
             reinterpret_cast<uint32_t*>(ws.cscore), ws.chi, sel, nsel, ws.header, tc ? 1 : 0};
  const size_t smem = sizeof(int32_t) * kCandCap * 2 + sizeof(float) * (kScoreMaxHeads * 128 + kScoreMaxHeads);
  cudaError_t err = cudaFuncSetAttribute(k7_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  k7_topk<<<d.L * d.R, kTopkThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsmoe
