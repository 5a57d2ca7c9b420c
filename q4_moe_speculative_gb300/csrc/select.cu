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
#include "common.cuh"
#include "kernels.h"

namespace dsmoe {
namespace {

constexpr int kCompactThreads = 1024;
constexpr int kScoreThreads = 128;   // one key per thread, one tile of keys per CTA
constexpr int kScoreMaxHeads = 16;
constexpr int kTopkThreads = 1024;
constexpr int kResidCap = 4096;      // residual bucket kept in shared memory

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

// ---------------------------------------------------------------------------------
// K5: canonical scoring of admitted blocks. CTA = (layer, 128 consecutive blocks); a
// key is loaded only if some row admits it, once for all rows. For each admitted row:
//   d_h = fmaf chain over i ascending (q_h[i] * k[i]) from 0.0f,
//   s = fmaf chain over h ascending (w_h * max(d_h, +0)) from +0.0f,
// written to the row's compacted position (word offset + rank within the word).
// ---------------------------------------------------------------------------------
struct ScoreArgs {
  int L, R, Hh, N;
  int64_t key_stride;
  const uint16_t* keys;
  const uint16_t* q;
  const float* hw;
  const uint32_t* mask;
  const int32_t* limit;
  const int32_t* wordoff;
  float* cscore;
};

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

  uint32_t rows = 0;
  if (b < a.N) {
    for (int r = 0; r < R; ++r) {
      const size_t lr = (size_t)l * R + r;
      int lim = a.limit[lr];
      if (b < lim && ((a.mask[lr * W + (b >> 5)] >> (b & 31)) & 1u)) rows |= 1u << r;
    }
  }
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
    const int wi = b >> 5;
    const uint32_t mw = admitted_word(a.mask + lr * W, wi, a.limit[lr]);
    const int pos = a.wordoff[lr * W + wi] + __popc(mw & ((1u << (b & 31)) - 1u));
    a.cscore[lr * (size_t)a.N + pos] = s;
  }
}

// Order-preserving 32-bit key of an fp32 score: larger score -> larger key, -0 == +0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------------
// K7: bounded radix top-k per (layer, row). Two 8-bit histogram passes over the
// compacted scores narrow the k-th largest key to a 16-bit prefix; the elements of that
// bucket are gathered into shared memory (bounded; above the bound the passes continue
// over global memory) and the last 16 bits are resolved there. The output pass walks the
// compacted array in order and takes every key above the threshold plus the first
// `need` keys equal to it, i.e. the lowest block indices among equal scores.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kTopkThreads)
    k7_topk(int N, int K, const int32_t* __restrict__ cidx, const int32_t* __restrict__ ccount,
            const float* __restrict__ cscore, int32_t* __restrict__ sel,
            int32_t* __restrict__ nsel, uint32_t* status) {
  __shared__ int hist[256];
  __shared__ int scratch[33];
  __shared__ int s_bucket, s_need;
  __shared__ uint32_t r_key[kResidCap];
  __shared__ int s_rn;

  const int lr = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = ccount[lr];
  const int32_t* ci = cidx + (size_t)lr * N;
  const float* cs = cscore + (size_t)lr * N;
  int32_t* out = sel + (size_t)lr * K;

  if (n <= K) {
    for (int i = tid; i < K; i += blockDim.x) out[i] = i < n ? ci[i] : -1;
    if (tid == 0) nsel[lr] = n;
    return;
  }

  uint32_t prefix = 0;
  int need = K;
  bool resid_in_smem = false;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    if (resid_in_smem) {
      const int rn = s_rn < kResidCap ? s_rn : kResidCap;
      for (int i = tid; i < rn; i += blockDim.x) {
        const uint32_t key = r_key[i];
        if ((key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
    } else {
      for (int i = tid; i < n; i += blockDim.x) {
        const uint32_t key = score_key(cs[i]);
        if (pass == 0 || (key >> (shift + 8)) == prefix)
          atomicAdd(&hist[(key >> shift) & 255], 1);
      }
    }
    __syncthreads();
    // Bucket holding the need-th largest: suffix counts from the top bucket down.
    if (tid == 0) {
      s_bucket = -1;
      s_need = need;
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
      if (tid == 0) flag_status(status, kStatusCheck);
      if (tid == 0) s_bucket = 0;
      __syncthreads();
    }
    prefix = (prefix << 8) | (uint32_t)s_bucket;
    need = s_need;
    if (pass == 1) {
      // Gather the 16-bit-prefix bucket (bounded) for the remaining two passes.
      const int cnt = hist[s_bucket];
      if (cnt <= kResidCap) {
        if (tid == 0) s_rn = 0;
        __syncthreads();
        for (int i = tid; i < n; i += blockDim.x) {
          const uint32_t key = score_key(cs[i]);
          if ((key >> 16) == prefix) {
            const int p = atomicAdd(&s_rn, 1);
            if (p < kResidCap) r_key[p] = key;
          }
        }
        __syncthreads();
        resid_in_smem = true;
        if (s_rn != cnt && tid == 0) flag_status(status, kStatusCheck);
      }
    }
    __syncthreads();
  }
  const uint32_t T = prefix;

  int taken = 0, eq_seen = 0;
  for (int c0 = 0; c0 < n && taken < K; c0 += blockDim.x) {
    const int i = c0 + tid;
    uint32_t key = 0;
    if (i < n) key = score_key(cs[i]);
    const int gt = (i < n) && key > T;
    const int eq = (i < n) && key == T;
    int eq_total;
    const int eq_rank = eq_seen + block_excl_scan(eq, scratch, &eq_total);
    const int take = gt || (eq && eq_rank < need);
    int take_total;
    const int pos = taken + block_excl_scan(take, scratch, &take_total);
    if (take && pos < K) out[pos] = ci[i];
    taken += take_total;
    eq_seen += eq_total;
  }
  if (tid == 0) {
    nsel[lr] = K;
    if (taken != K) flag_status(status, kStatusCheck);
  }
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
  L.total = off;
  return L;
}

cudaError_t launch_compact(const SelDims& d, const uint32_t* mask, const int32_t* limit,
                           const SelWorkspace& ws, cudaStream_t s) {
  k6_compact<<<d.L * d.R, kCompactThreads, 0, s>>>(d.R, d.N, mask, limit, ws.wordoff, ws.cidx,
                                                   ws.ccount);
  return cudaGetLastError();
}

cudaError_t launch_score(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                         const float* head_w, const uint32_t* mask, const int32_t* limit,
                         const SelWorkspace& ws, cudaStream_t s) {
  const int RH = d.R * d.Hh;
  const size_t smem = sizeof(float) * ((size_t)RH * 128 + ((RH + 3) & ~3)) +
                      (size_t)kScoreThreads * 16 * sizeof(uint4);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(k5_score, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
  }
  const int tiles = (d.N + kScoreThreads - 1) / kScoreThreads;
  ScoreArgs a{d.L, d.R, d.Hh, d.N, d.key_stride, keys, q, head_w, mask, limit, ws.wordoff,
              ws.cscore};
  k5_score<<<d.L * tiles, kScoreThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_topk(const SelDims& d, int32_t* sel, int32_t* nsel, const SelWorkspace& ws,
                        cudaStream_t s) {
  k7_topk<<<d.L * d.R, kTopkThreads, 0, s>>>(d.N, d.topk, ws.cidx, ws.ccount, ws.cscore, sel,
                                             nsel, ws.header);
  return cudaGetLastError();
}

}  // namespace dsmoe
