// select.cu — compressed-attention block selection: compaction of the admitted index
// (K6), scoring of admitted blocks only (K5) and the bounded radix top-k (K7).
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)",
// paragraph "Decode at depth": compressed attention picks 512 blocks per layer; layers
// score only the blocks their mask admits, compact the admitted index once per row and
// select the top 512 with a bounded radix select.
//
// Chain on the device:
//  K6  per (layer, row): the admitted index of the row (ascending, written once) and its
//      count; per layer: the union of the rows' admitted blocks ("union list", ascending)
//      with, for each entry, the rows that admit it.
//  K5  scores every union entry for the rows that admit it; results are stored by union
//      position [layer][row][entry]. Rows that do not admit an entry get a sentinel that
//      sorts below every score.
//  K7  per (layer, row): bounded radix top-k over the union entries, in one CTA (tensor-core
//      mode: a collection threshold from per-chunk maxima, collection, candidates, canonical
//      re-score of the uncertain ones, final select).
//
// Two scoring modes give the same selection:
//  * canonical: every score in the canonical fp32 order (fmaf over i ascending, then over
//    heads ascending) on CUDA cores;
//  * tensor-core (default): q_h . k for a tile of 128 union keys as one
//    [128 x 128] x [128 x R*Hh] bf16 contraction on tcgen05 (keys gathered by cp.async into
//    the 128-byte swizzled K-major layout, queries likewise, fp32 accumulators in TMEM),
//    giving an interval [lo, hi] that contains the canonical score:
//    |s_tc - s_canon| <= eps = 2^-13 * ||k|| * sum_h |w_h| ||q_h||. Both dot products are
//    sums of 128 exact products whose magnitudes add up to at most ||q_h|| ||k||: the
//    canonical chain rounds 128 times (at most 2^-17 of that sum); the tensor core adds 8
//    groups of 16 products to an fp32 accumulator, and even 16 units in the last place of
//    that sum per group (far more than the hardware loses) stay below 2^-16 of it. The
//    two sums over the heads add 2 x 8 roundings of terms below |w_h| ||q_h|| ||k|| (2^-20).
//    In all at most 2^-15.2 of ||k|| sum_h |w_h| ||q_h||, so 2^-13 leaves a margin above 4.
//    K5 stores s_tc per admitting row and ||k|| per entry (and, per 32 entries, the largest
//    ||k|| and each row's largest s_tc); every consumer derives [lo, hi]
//    with the same function (tc_lo / tc_hi), so the bounds agree bit for bit. K7 takes
//    T = k-th largest lo; every block of the canonical top-k has hi >= T, so only the
//    candidates with hi >= T are re-scored in the canonical order and selected among
//    exactly. The result is identical to the canonical mode by construction.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace dsmoe {
namespace {

constexpr int kCompactThreads = 512;   // 3 CTAs per SM
constexpr int kScoreThreads = 128;   // canonical scorer: one key per thread
constexpr int kScoreMaxHeads = 16;
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kResidCap = 4096;      // residual radix bucket kept in shared memory
constexpr int kCandCap = 4096;       // re-score candidates kept in shared memory
constexpr int kCollectCap = 4096;    // entries the threshold-tau collection keeps
constexpr uint32_t kWaitPolls = 1u << 17;   // bounded mbarrier polling (<= ~0.13 s)
constexpr float kEpsRel = 0.0001220703125f;  // 2^-13
constexpr uint32_t kNoScoreKey = 0u;        // sorts below the key of every score
constexpr uint32_t kMinusInfBits = 0xFF800000u;

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

// Admitted bits of mask word wi for a row with limit lim (bits at b >= lim cleared). The
// load is predicated rather than branched around, so that a thread's loads of several
// words and rows are all in flight together.
__device__ __forceinline__ uint32_t admitted_word(const uint32_t* m, int wi, int lim) {
  const int rem = lim - wi * 32;
  const uint32_t w = rem > 0 ? __ldg(m + wi) : 0u;
  return rem >= 32 ? w : (rem > 0 ? w & ((1u << rem) - 1u) : 0u);
}

// d0 + qa k, d1 + qb k for the bf16 pair (qa, qb) of qw and the bf16 k in the low (HI =
// false) or high half of kw: fused multiply-adds of bf16 operands into fp32 (exact
// product, one rounding), the same values as fmaf on the operands widened to fp32.
template <bool HI>
__device__ __forceinline__ void fma_pair_bf16(float& d0, float& d1, uint32_t qw, uint32_t kw) {
  if (HI)
    asm("{\n\t.reg .b16 qa, qb, kl, kh;\n\t"
        "mov.b32 {qa, qb}, %2;\n\tmov.b32 {kl, kh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, qa, kh, %0;\n\tfma.rn.f32.bf16 %1, qb, kh, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(qw), "r"(kw));
  else
    asm("{\n\t.reg .b16 qa, qb, kl, kh;\n\t"
        "mov.b32 {qa, qb}, %2;\n\tmov.b32 {kl, kh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, qa, kl, %0;\n\tfma.rn.f32.bf16 %1, qb, kl, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(qw), "r"(kw));
}

// d + q_lo k_lo, then + q_hi k_hi, for two packed bf16 pairs: each step is one fused
// multiply-add of bf16 operands into fp32 (the product is exact, one rounding), the same
// value as fmaf on the operands widened to fp32.
__device__ __forceinline__ float fma2_bf16(uint32_t qw, uint32_t kw, float d) {
  asm("{\n\t.reg .b16 ql, qh, kl, kh;\n\t"
      "mov.b32 {ql, qh}, %1;\n\tmov.b32 {kl, kh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ql, kl, %0;\n\tfma.rn.f32.bf16 %0, qh, kh, %0;\n\t}"
      : "+f"(d)
      : "r"(qw), "r"(kw));
  return d;
}

// Order-preserving 32-bit key of an fp32 score: larger score -> larger key, -0 == +0.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The fp32 score of an order-preserving key (inverse of score_key; -0 comes back as +0).
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr uint32_t kCertainKey = 0xFFFFFFFFu;   // above the key of every finite score

// Interval [lo, hi] (order keys) around a tensor-core score s (fp32 bits) that contains the
// canonical score: eps = kn * G rounded upward (kn the key norm bound, G the row's
// 2^-13 * sum_h |w_h| ||q_h|| rounded upward), lo = s - eps rounded downward, hi = s + eps
// rounded upward. An entry the row does not admit (s = -inf) gets lo = kNoScoreKey and
// hi = the key of -inf.
__device__ __forceinline__ uint32_t tc_lo(uint32_t sbits, float kn, float G) {
  if (sbits == kMinusInfBits) return kNoScoreKey;
  return score_key(__fsub_rd(__uint_as_float(sbits), __fmul_ru(kn, G)));
}
__device__ __forceinline__ uint32_t tc_hi(uint32_t sbits, float kn, float G) {
  if (sbits == kMinusInfBits) return score_key(__uint_as_float(kMinusInfBits));
  return score_key(__fadd_ru(__uint_as_float(sbits), __fmul_ru(kn, G)));
}

// Max over the warp of eight values per lane, reduce-scatter style (nine shuffles): lane L
// ends with the maximum of value 4 b4 + 2 b3 + b2 (b = the bits of L) over all lanes.
__device__ __forceinline__ float warp_max8(const float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  float a[4], b[2];
  const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
#pragma unroll
  for (int j = 0; j < 4; ++j)   // keep values 4 h4 + j, send the partner's half
    a[j] = fmaxf(h4 ? v[4 + j] : v[j], __shfl_xor_sync(0xffffffffu, h4 ? v[j] : v[4 + j], 16));
#pragma unroll
  for (int j = 0; j < 2; ++j)
    b[j] = fmaxf(h3 ? a[2 + j] : a[j], __shfl_xor_sync(0xffffffffu, h3 ? a[j] : a[2 + j], 8));
  float c = fmaxf(h2 ? b[1] : b[0], __shfl_xor_sync(0xffffffffu, h2 ? b[0] : b[1], 4));
  c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 2));
  return fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 1));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Place of head h among the kScoreMaxHeads query values of one element in the fp32 query
// layout of the top-k: heads h = 4j + t at t * 4 + j, so that thread t of a candidate's four
// reads the values of its heads t, t + 4, t + 8, t + 12 as one 16-byte word.
__host__ __device__ constexpr int qslot(int h) { return (h & 3) * 4 + (h >> 2); }

// Canonical score of one block: q fp32 (shared) in the layout [i][kScoreMaxHeads] (value i
// of head h at i * kScoreMaxHeads + qslot(h)), key 128 bf16 (global), w [Hh].
__device__ __forceinline__ float canonical_score(const float* q, const uint16_t* key,
                                                 const float* w, int Hh) {
  float d[kScoreMaxHeads];
#pragma unroll
  for (int h = 0; h < kScoreMaxHeads; ++h) d[h] = 0.0f;
  const uint4* k4 = reinterpret_cast<const uint4*>(key);
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint4 kvs[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) kvs[c] = __ldg(k4 + half * 8 + c);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      const uint4 kv = kvs[c];
      const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                           bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
      for (int h = 0; h < kScoreMaxHeads; ++h) {
        if (h < Hh) {
          const float* qh = q + ((half * 8 + c) * 8) * kScoreMaxHeads + qslot(h);
          float t = d[h];
#pragma unroll
          for (int e = 0; e < 8; ++e) t = __fmaf_rn(qh[e * kScoreMaxHeads], kf[e], t);
          d[h] = t;
        }
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
// K6: compaction. CTAs [0, L*R): one per (layer, row): popcount + block scan of the
// admitted words, then each warp scatters the admitted indices of 32 words with a ballot
// over per-lane predicates (bit set and block below the causal limit). CTAs [L*R, L*R+L):
// one per layer: the same over the union of the rows' admitted words, recording for each
// union entry the rows that admit it, plus each union word's exclusive offset. A row CTA
// counts first and scatters only when its compacted index is wanted: when the caller
// asked for it, or when the row admits at most top_k blocks (the top-k then copies it).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct CompactArgs {
  int L, R, N;
  const uint32_t* mask;
  const int32_t* limit;
  int32_t* cidx;
  int32_t* ccount;
  int32_t* uidx;       // [L][N]
  int32_t* ucount;     // [L]
  uint8_t* urows;      // [L][N]
  int32_t* uwordoff;   // [L][W]
  uint32_t* uagg;      // [L][P] published union counts of the chunks
  uint32_t* status;
  int topk;
  int want_cidx;       // the caller passed cidx / ccount
};

__global__ void __launch_bounds__(kCompactThreads, 3) k6_compact(CompactArgs a) {
  pdl_trigger();   // the scorer may launch as soon as every CTA of this grid has started
  __shared__ int scratch[33];
  __shared__ int s_base;
  const int R = a.R, N = a.N;
  const int W = (N + 31) >> 5;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // union CTAs (the longer ones, first): one per (layer, chunk of kCompactThreads words);
  // then one row CTA per (layer, row)
  const int P = (W + kCompactThreads - 1) / kCompactThreads;
  const bool union_cta = (int)blockIdx.x < a.L * P;
  const int uc = blockIdx.x;
  const int lr = (int)blockIdx.x - a.L * P;   // meaningful for row CTAs only
  const int l = union_cta ? uc / P : lr / R;
  const int uchunk = union_cta ? uc - l * P : 0;
  const uint32_t* mrow = a.mask + (size_t)(union_cta ? l * R : lr) * W;
  // the rows' causal limits, read by every thread (no barrier before the mask loads); a
  // word's bits at or past the limit are cleared after it is loaded
  int lims[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int lim = r < R ? __ldg(a.limit + (size_t)l * R + r) : 0;
    lims[r] = lim < 0 ? 0 : (lim > N ? N : lim);
  }
  const int lim_row = union_cta ? 0 : min(max(__ldg(a.limit + lr), 0), N);
  auto limited = [](uint32_t w, int wi, int lim) {
    const int rem = lim - wi * 32;
    return rem >= 32 ? w : (rem > 0 ? w & ((1u << rem) - 1u) : 0u);
  };

  if (!union_cta && !a.want_cidx) {
    int c = 0;
    for (int wi = tid; wi < W; wi += kCompactThreads) c += __popc(admitted_word(mrow, wi, lim_row));
    int total;
    block_excl_scan(c, scratch, &total);
    if (total > a.topk) {
      if (tid == 0) a.ccount[lr] = total;
      return;
    }
  }

  int base = 0;
  int c_first = 0, c_last = W;
  if (union_cta) {   // this CTA's chunk (one pass of the loop below)
    c_first = uchunk * kCompactThreads;
    c_last = min(W, c_first + kCompactThreads);
  }
  for (int c0 = c_first; c0 < c_last; c0 += kCompactThreads) {
    // word wi = c0 + tid of each row read (per row for the union): its admitted bits
    const int wi = c0 + tid;
    uint32_t mine[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) mine[r] = 0u;
    if (wi < W) {
      if (union_cta) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < R) mine[r] = __ldg(a.mask + ((size_t)l * R + r) * W + wi);
#pragma unroll
        for (int r = 0; r < 8; ++r) mine[r] = limited(mine[r], wi, lims[r]);
      } else {
        mine[0] = admitted_word(mrow, wi, lim_row);
      }
    }
    uint32_t mw = 0;
#pragma unroll
    for (int r = 0; r < 8; ++r) mw |= mine[r];
    // a word whose admitted bits are the same in every row (a shared mask away from the
    // limits): each of its union entries is admitted by every row
    bool same = true;
#pragma unroll
    for (int r = 1; r < 8; ++r)
      if (r < R) same = same && mine[r] == mine[0];
    int total;
    const int lexcl = block_excl_scan(__popc(mw), scratch, &total);
    if (union_cta) {
      // publish this chunk's count, then add up those of the chunks before it in the
      // layer: lower block indices, started earlier, and none of them waits on this one
      uint32_t* agg = a.uagg + (size_t)l * P;
      if (tid == 0) {
        __threadfence();
        atomicExch(agg + uchunk, 0x80000000u | (uint32_t)total);
      }
      if (warp == 0) {
        int v = 0;
        for (int j = lane; j < uchunk; j += 32) {
          uint32_t x = 0;
          for (uint32_t it = 0; it < (1u << 22); ++it) {
            x = ld_acquire_u32(agg + j);
            if (x & 0x80000000u) break;
            __nanosleep(64);
          }
          if (!(x & 0x80000000u)) flag_status(a.status, kStatusTimeout);
          v += (int)(x & 0x7FFFFFFFu);
        }
        v = __reduce_add_sync(0xffffffffu, v);
        if (lane == 0) s_base = v;
      }
      __syncthreads();
      base = s_base;
    }
    const int excl = base + lexcl;
    if (union_cta && wi < W) a.uwordoff[(size_t)l * W + wi] = excl;
    // Warp `warp` scatters the words c0 + 32*warp .. c0 + 32*warp + 31 of this chunk, whose
    // bits and offsets sit in its lanes 0..31, one word at a time, broadcast by shuffles
    // (nothing goes through shared memory, so the words' stores overlap).
    {
      const int wbase = c0 + warp * 32;
      const uint32_t all_rows = (1u << R) - 1u;
      const int nw = min(32, W - wbase);
      int32_t* const uo = a.uidx + (size_t)l * N;
      uint8_t* const ro = a.urows + (size_t)l * N;
      int32_t* const co = union_cta ? nullptr : a.cidx + (size_t)lr * N;
#pragma unroll 4
      for (int jw = 0; jw < nw; ++jw) {
        const int w = wbase + jw;
        const int b = w * 32 + lane;
        const uint32_t wv = __shfl_sync(0xffffffffu, mw, jw);
        const int off0 = __shfl_sync(0xffffffffu, excl, jw);
        const bool pred = (wv >> lane) & 1u;
        uint32_t rows = 0;
        if (union_cta) {
          if (__shfl_sync(0xffffffffu, same ? 1 : 0, jw)) {
            rows = pred ? all_rows : 0u;
          } else {
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < R && ((__shfl_sync(0xffffffffu, mine[r], jw) >> lane) & 1u)) rows |= 1u << r;
          }
        }
        if (pred) {
          const int off = off0 + __popc(wv & ((1u << lane) - 1u));
          if (union_cta) {
            uo[off] = b;
            ro[off] = (uint8_t)rows;
          } else {
            co[off] = b;
          }
        }
      }
    }
    base += total;
    __syncthreads();
  }
  if (tid == 0) {
    if (!union_cta) a.ccount[lr] = base;
    else if (c_last == W) a.ucount[l] = base;
  }
}

struct ScoreArgs {
  int L, R, Hh, N;
  int64_t key_stride;
  const uint16_t* keys;
  const uint16_t* q;
  const float* hw;
  const uint32_t* mask;
  const int32_t* limit;
  const int32_t* uidx;
  const int32_t* ucount;
  const uint8_t* urows;
  const int32_t* uwordoff;
  uint32_t* sc0;      // [L][R][NS] by union entry: fp32 scores (-inf: not admitted)
  float* knorm;       // [L][NS] by union entry: key norm bound (tensor-core mode)
  float* qnorm;       // [L][R] 2^-13 sum_h |w_h| ||q_h|| bound (tensor-core mode)
  float* kmax;        // [L][NC] the largest knorm of each 32 union entries (tensor-core mode)
  uint32_t* status;
  int tma;            // kmap is valid: tiles of 128 consecutive blocks come by TMA
  CUtensorMap kmap;   // keys [L][N][128] bf16, boxes of 64 values x 128 blocks, 128B swizzle
  int NS;             // row stride of sc0 / knorm (N rounded up to a multiple of 4)
  int NC;             // row stride of kmax
  float* smax;        // [L][NC][R] per 32 union entries, each row's largest score
                      // (-inf: none admitted; tensor-core mode)
};

// ---------------------------------------------------------------------------------
// K5 (canonical mode): CUDA-core scoring. CTA = (layer, 128 consecutive blocks); a key
// is loaded only if some row admits it, once for all rows; scores go to the key's union
// position; rows that do not admit it get -inf there.
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

  uint32_t rows = 0, uw = 0;
  if (b < a.N) {
    for (int r = 0; r < R; ++r) {
      const size_t lr = (size_t)l * R + r;
      const uint32_t m = admitted_word(a.mask + lr * W, b >> 5, a.limit[lr]);
      uw |= m;
      if ((m >> (b & 31)) & 1u) rows |= 1u << r;
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
  const int e = a.uwordoff[(size_t)l * W + (b >> 5)] + __popc(uw & ((1u << (b & 31)) - 1u));

  for (int r = 0; r < R; ++r) {
    const size_t out = ((size_t)l * R + r) * a.NS + e;
    if (!(rows & (1u << r))) {
      a.sc0[out] = kMinusInfBits;
      continue;
    }
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
    a.sc0[out] = __float_as_uint(s);
  }
}

// 16-byte async copy global -> shared; zero-fill (no global read) when !valid.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

// The same with an L2 eviction-priority hint: streamed data (read once) goes first, so that
// the scores written meanwhile stay in L2 for the top-k that reads them next.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Scores and key norms written by K5 are read back by K7 right after: kept in L2 ahead of
// the streamed keys, then read with evict_first so that they leave first once read.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_hint(uint32_t* p, uint32_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void st_hint(float* p, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint4 ld_hint_v4(const uint32_t* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, bool valid,
                                                uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint.L2::256B [%0], [%1], 16, %2, %3;" ::"r"(dst),
               "l"(src), "r"(valid ? 16 : 0), "l"(policy)
               : "memory");
}

// ---------------------------------------------------------------------------------
// K5 (tensor-core mode): one persistent CTA per SM scores a contiguous range of the
// layers' union tiles (128 union entries each). Roles:
//  * four producer warps fill a ring of kStages stage buffers with each tile's keys in the
//    128-byte swizzled K-major layout (row r's 16-byte chunk j of each 64-value half at
//    r*128 + ((j ^ (r & 7)) * 16)). A tile of 128 consecutive block ids (the common case:
//    the union of the rows' admitted blocks is dense) is two TMA boxes of 64 values x 128
//    blocks that the copy engine swizzles; any other tile is gathered with 16-byte
//    cp.async, published on the stage's `full` barrier once the warp's copies have landed
//    (cp.async.wait_group, then a proxy fence), kLag tiles behind the newest one. The
//    block ids, entry count and row masks of the next tile are loaded while the current
//    one is issued; the tile's layer, first entry, count and row masks go to shared
//    memory beside the stage, so the epilogue reads nothing from global memory. Producer
//    warp 0 also stages each layer's queries (one of two slots, by layer parity) with their
//    norm bounds and head weights;
//  * three epilogue groups of 4 warps (two when N > 64) take the tiles in turn; each has
//    its own TMEM accumulator. The group's first thread issues the 8 tcgen05.mma (M = 128 keys,
//    N = NPAD >= R*Hh, K = 16 each) and commits to the group's mbarrier; each warp then
//    reads its 32 lanes (one key per thread), writes the score for every admitting row and
//    the key's norm bound, and releases the stage on its `empty` barrier.
// Waits are bounded; a give-up sets DS_ERR_TIMEOUT in the status word and an abort flag
// that every role checks before its next wait; the group that issued MMAs waits once more
// (bounded) for them before TMEM is freed.
// ---------------------------------------------------------------------------------
constexpr int kTcProducerWarps = 4;
constexpr int kTcRowsPerProducer = 128 / kTcProducerWarps;   // 32: one block id per lane

template <int NCH>
struct TcGeom {
  static constexpr int NPAD = NCH * 16;
  static constexpr uint32_t kCols = NPAD <= 32 ? 32 : (NPAD <= 64 ? 64 : 128);  // per group
  // epilogue groups of 4 warps, each with its own accumulator: three while the epilogue's
  // registers fit 512 threads (N <= 64), else two
  static constexpr int kGroups = NPAD <= 64 ? 3 : 2;
  static constexpr int kThreads = 32 * (kTcProducerWarps + 4 * kGroups);
  static constexpr uint32_t kKeyBytes = 128 * 256;   // one tile of keys
  static constexpr uint32_t kQBytes = NPAD * 256;    // one layer's queries
  static constexpr int kFit = (int)((227u * 1024u - 4096u - 2u * kQBytes) / kKeyBytes);
  static constexpr int kStages = kFit < 6 ? kFit : 6;
  static constexpr int kLag = kStages - kGroups;     // tiles in flight behind the newest
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kKeyBytes + 2 * (size_t)kQBytes;
  static_assert(kLag >= 1, "stage ring too small");
  // tcgen05.alloc takes a power of two of at least 32 columns
  static constexpr uint32_t kTmemCols =
      kGroups * kCols <= 128 ? 128 : (kGroups * kCols <= 256 ? 256 : 512);
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "TMEM allocation must be a power of two");
};

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sm100::smem_u32(bar)) : "memory");
}
// Barrier `id` over `n` threads that also returns whether `pred` held in all of them.
__device__ __forceinline__ bool bar_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Tile t of the layers' union tiles (128 entries each, empty layers skipped): its layer and
// first entry; *total gets the number of tiles. Warp-cooperative, every lane gets the result.
__device__ __forceinline__ void tile_cursor(const int32_t* ucount, int L, int t, int* l_out,
                                            int* e_out, int* total) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  *l_out = L;
  *e_out = 0;
  bool found = false;
  for (int l0 = 0; l0 < L; l0 += 32) {
    const int l = l0 + lane;
    const int nt = l < L ? (ucount[l] + 127) >> 7 : 0;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, carry + incl > t);
    if (!found && hit) {
      const int src = __ffs(hit) - 1;
      const int excl = __shfl_sync(0xffffffffu, incl - nt, src);
      *l_out = l0 + src;
      *e_out = (t - carry - excl) * 128;
      found = true;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  *total = carry;
}

template <int NCH, int HH>
__global__ void __launch_bounds__(TcGeom<NCH>::kThreads, 1) k5_score_tc(const __grid_constant__ ScoreArgs a) {
  using G = TcGeom<NCH>;
  constexpr int NPAD = G::NPAD, S = G::kStages, D = G::kLag;
  constexpr uint32_t kCols = G::kCols, kKeyBytes = G::kKeyBytes, kQBytes = G::kQBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[S];
  __shared__ __align__(8) uint64_t bar_empty[S];
  __shared__ __align__(8) uint64_t bar_mma[G::kGroups];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_w[2][NPAD];
  __shared__ float s_wg[G::kGroups][NPAD];      // each epilogue group's copy of its layer's w
  __shared__ float s_F[2][8];
  __shared__ float s_qn[NPAD];
  __shared__ int s_tl[S], s_te[S], s_tn[S];     // per stage: layer, first entry, entry count
  __shared__ uint8_t s_trows[S][128];           // per stage: row masks of the 128 entries

  const int R = a.R, Hh = a.Hh, RH = R * Hh, N = a.N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const uint32_t raw = sm100::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t qslot_addr = base + (uint32_t)S * kKeyBytes;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      sm100::mbar_init(&bar_full[s], kTcProducerWarps);
      sm100::mbar_init(&bar_empty[s], 4);
    }
    for (int g = 0; g < G::kGroups; ++g) sm100::mbar_init(&bar_mma[g], 1);
    s_abort = 0;
    sm100::fence_mbar_init();
  }
  if (warp == 0) {
    sm100::tmem_alloc(&s_tmem, G::kTmemCols);
    sm100::tmem_relinquish();
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = s_tmem;

  // Set up while the compaction finishes (programmatic launch); its union lists and counts
  // are read from here on.
  pdl_wait();
  pdl_trigger();   // the top-k may start launching on SMs this grid leaves
  // This CTA's tile range [t0, t1) and the cursor of t0 (same in every warp).
  int total = 0, cl = 0, ce = 0;
  tile_cursor(a.ucount, a.L, 0, &cl, &ce, &total);
  const int t0 = (int)(((long long)blockIdx.x * total) / gridDim.x);
  const int t1 = (int)(((long long)(blockIdx.x + 1) * total) / gridDim.x);
  if (t0 >= t1) {
    if (warp == 0) sm100::tmem_dealloc(tmem, G::kTmemCols);
    return;
  }
  if (t0 > 0) tile_cursor(a.ucount, a.L, t0, &cl, &ce, &total);
  const int n = t1 - t0;

  auto give_up = [&]() {
    if (lane == 0) {
      s_abort = 1;
      flag_status(a.status, kStatusTimeout);
    }
  };

  if (warp < kTcProducerWarps) {
    // ------------------------------------------------------------- producers -----
    const int pw = warp;
    const uint64_t kpol = l2_evict_first_policy();   // keys are read once
    int l = cl, e0 = ce;
    int lcnt = a.ucount[cl];    // entry count of layer l
    int qlayer[2] = {-1, -1};   // layer staged in each query slot
    int qlast[2] = {-1, -1};    // last tile (local index) that reads each slot
    int pub = 0;                // next tile to publish on its full barrier
    uint32_t tma_bits = 0;      // bit (j & 31): tile j came by TMA (its arrivals are done)
    auto publish = [&](int last) {   // gathered tiles pub..last, whose copies have landed
      fence_proxy_async();
      __syncwarp();
      if (lane == 0)
        for (int j = pub; j <= last; ++j)
          if (!((tma_bits >> (j & 31)) & 1u)) mbar_arrive1(&bar_full[j % S]);
      pub = last + 1;
    };
    auto pwait = [&](uint64_t* bar, uint32_t parity) {   // warp-uniform bounded wait
      return __all_sync(0xffffffffu, sm100::mbar_wait(bar, parity, kWaitPolls));
    };
    // Next tile after (lcur, ecur) of a layer with cnt entries; empty layers are skipped.
    auto padvance = [&](int& lcur, int& ecur, int& cnt) {
      ecur += 128;
      if (ecur >= cnt) {
        ecur = 0;
        for (++lcur; lcur < a.L; ++lcur)
          if ((cnt = a.ucount[lcur]) > 0) break;
      }
    };
    // What the tile at (ll, ee) needs from global memory, loaded one tile ahead and not
    // touched until that tile is issued: the block id of this warp's row `lane`, the first
    // and last block ids (a tile of 128 consecutive blocks is one TMA box pair) and, in
    // warp 0, the row masks of the tile's entries ee + lane + 32k.
    struct Pref {
      int ucnt, id, bf, bl;
      uint32_t rw[4];
    };
    auto prefetch = [&](int ll, int ee, int cnt, Pref& p) {
      p.ucnt = cnt;
      const int32_t* u = a.uidx + (size_t)ll * N;
      const int r0 = ee + pw * kTcRowsPerProducer + lane;
      p.id = r0 < cnt ? u[r0] : 0;
      p.bf = u[ee];
      p.bl = ee + 127 < cnt ? u[ee + 127] : -1;
      const uint8_t* ur = a.urows + (size_t)ll * N;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = ee + lane + 32 * k;
        p.rw[k] = (pw == 0 && e < cnt) ? (uint32_t)ur[e] : 0u;
      }
    };
    // One tile: `cur` holds its prefetched indices, `nxt` receives the next tile's. The
    // loop below alternates two of these so that no copy waits for a load in flight.
    auto step = [&](int i, const Pref& cur, Pref& nxt) -> bool {
        const int s = i % S;
        {  // the next tile's indices, in flight while this one is issued
          int ln = l, en = e0, cn = lcnt;
          padvance(ln, en, cn);
          if (i + 1 < n) prefetch(ln, en, cn, nxt);
        }
        if (s_abort) return false;
        if (i >= S && !pwait(&bar_empty[s], ((i / S) - 1) & 1)) {
          give_up();
          return false;
        }
        const int slot = l & 1;
        if (qlayer[slot] != l) {
          // every tile issued so far is published, then (warp 0) the slot's readers drain
          if (pub < i) {
            cp_async_wait<0>();
            publish(i - 1);
          }
          if (pw == 0) {
            for (int u = (i - S + 1 > 0 ? i - S + 1 : 0); u <= qlast[slot]; ++u)
              if (!pwait(&bar_empty[u % S], (u / S) & 1)) {
                give_up();
                return false;
              }
            // queries of layer l (rows >= R*Hh are zero) in the swizzled K-major layout, all
            // copies in flight at once, then their norm bounds, the weights and F_r
            const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(a.q + (size_t)l * RH * 128);
            const uint32_t qa = qslot_addr + (uint32_t)slot * kQBytes;
            for (int idx = lane; idx < NPAD * 16; idx += 32) {
              const int p = idx >> 4, c = idx & 15;
              const uint32_t dst = qa + (uint32_t)(c >> 3) * (kQBytes / 2) + (uint32_t)p * 128u +
                                   (uint32_t)(((c & 7) ^ (p & 7)) << 4);
              cp_async16(dst, qsrc + (size_t)(p < RH ? p : 0) * 256 + c * 16, p < RH);
            }
            cp_async_commit();
            cp_async_wait<0>();     // no tile's copies are outstanding here
            __syncwarp();
            const uint8_t* qp = base_ptr + (size_t)S * kKeyBytes + (size_t)slot * kQBytes;
            for (int p = lane; p < NPAD; p += 32) {
              // sum of squares rounded upward at every step: an upper bound of ||q_p||^2
              float ss = 0.0f;
#pragma unroll 4
              for (int c = 0; c < 16; ++c) {
                const uint4 v = *reinterpret_cast<const uint4*>(
                    qp + (c >> 3) * (kQBytes / 2) + p * 128 + (((c & 7) ^ (p & 7)) << 4));
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float lo = bf16_lo(wv[e]), hi = bf16_hi(wv[e]);
                  ss = __fmaf_ru(lo, lo, ss);
                  ss = __fmaf_ru(hi, hi, ss);
                }
              }
              s_qn[p] = __fmul_ru(__fsqrt_ru(ss), 1.0000153f);   // (1 + 2^-16) margin
            }
            for (int p = lane; p < NPAD; p += 32)
              s_w[slot][p] = p < RH ? a.hw[(size_t)l * RH + p] : 0.0f;
            __syncwarp();
            if (lane < R) {
              float F = 0.0f;
              for (int h = 0; h < Hh; ++h)
                F = __fmaf_ru(fabsf(s_w[slot][lane * Hh + h]), s_qn[lane * Hh + h], F);
              s_F[slot][lane] = F;
              a.qnorm[(size_t)l * R + lane] = __fmul_ru(kEpsRel, F);   // same from every CTA
            }
          }
          qlayer[slot] = l;
        }
        qlast[slot] = i;
        if (pw == 0) {   // the tile's layer, first entry, entry count and row masks
          if (lane == 0) {
            s_tl[s] = l;
            s_te[s] = e0;
            s_tn[s] = cur.ucnt;
          }
  #pragma unroll
          for (int k = 0; k < 4; ++k) s_trows[s][lane + 32 * k] = (uint8_t)cur.rw[k];
        }
        const bool boxed = a.tma != 0 && e0 + 128 <= cur.ucnt && cur.bl - cur.bf == 127;
        uint8_t* const sp = base_ptr + (size_t)s * kKeyBytes;
        if (boxed) {
          // 128 consecutive blocks: two boxes of 64 values x 128 blocks, swizzled by the copy
          tma_bits |= 1u << (i & 31);
          cp_async_commit();      // an empty group: one group per tile in either mode
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            if (pw == 0) {
              sm100::mbar_arrive_expect_tx(&bar_full[s], kKeyBytes);
              sm100::tma_load_3d(sp, &a.kmap, 0, cur.bf, l, &bar_full[s]);
              sm100::tma_load_3d(sp + kKeyBytes / 2, &a.kmap, 64, cur.bf, l, &bar_full[s]);
            } else {
              mbar_arrive1(&bar_full[s]);
            }
          }
        } else {
          // gather: this warp's 32 rows, two rows (512 contiguous bytes) per step
          tma_bits &= ~(1u << (i & 31));
          const uint8_t* kbase8 =
              reinterpret_cast<const uint8_t*>(a.keys + (size_t)l * a.key_stride);
          const uint32_t sa = base + (uint32_t)s * kKeyBytes;
#pragma unroll
          for (int jj = 0; jj < kTcRowsPerProducer / 2; ++jj) {
            const int rr = 2 * jj + (lane >> 4);
            const int r = pw * kTcRowsPerProducer + rr;
            const int c = lane & 15;
            const int b = __shfl_sync(0xffffffffu, cur.id, rr);
            const uint32_t dst = sa + (uint32_t)(c >> 3) * (kKeyBytes / 2) +
                                 (uint32_t)r * 128u + (uint32_t)(((c & 7) ^ (r & 7)) << 4);
            cp_async16_hint(dst, kbase8 + (size_t)b * 256 + c * 16, e0 + r < cur.ucnt, kpol);
          }
          cp_async_commit();
        }
        if (i - D >= pub) {
          cp_async_wait<D>();
          publish(i - D);
        }
        padvance(l, e0, lcnt);
        return true;
    };
    Pref pa, pb;
    prefetch(l, e0, lcnt, pa);
    bool ok = true;
    for (int i = 0; i < n && ok; i += 2) {
      ok = step(i, pa, pb);
      if (ok && i + 1 < n) ok = step(i + 1, pb, pa);
    }
    cp_async_wait<0>();
    if (ok && pub < n) publish(n - 1);
  } else {
    // ------------------------------------------------------------- epilogue ------
    const int g = (warp - kTcProducerWarps) >> 2;
    const int row = (warp & 3) * 32 + lane;          // TMEM lane = key row of the tile
    const bool leader = warp == kTcProducerWarps + 4 * g && lane == 0;
    const int bar_id = 1 + g;
    const uint32_t tbuf = tmem + (uint32_t)g * kCols;
    uint32_t mphase = 0;
    const uint64_t spol = l2_evict_last_policy();   // scores stay in L2 for K7
    bool issued = false;    // this group has MMAs whose commit it has not observed
    int wlayer = -1;        // layer whose head weights s_wg[g] holds
    for (int i = g; i < n; i += G::kGroups) {
      const int s = i % S;
      bool ok = !s_abort && sm100::mbar_wait(&bar_full[s], (i / S) & 1, kWaitPolls);
      ok = bar_and(bar_id, 128, ok);
      if (!ok) {
        if (warp == kTcProducerWarps + 4 * g) give_up();
        break;
      }
      const int l = s_tl[s], e0 = s_te[s], ucnt = s_tn[s];
      const int slot = l & 1;
      const uint32_t sa = base + (uint32_t)s * kKeyBytes;
      if (l != wlayer) {
        // the group's own copy of the head weights: the stage (and with it the query slot)
        // is released before the scores are formed, and the producer may then refill it
        const int t = (warp & 3) * 32 + lane;
        if (t < NPAD) s_wg[g][t] = s_w[slot][t];
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(128) : "memory");
        wlayer = l;
      }
      if (leader) {
        sm100::tc_fence_after();
        fence_proxy_async();
        constexpr uint32_t idesc = sm100::idesc_bf16_f32(128, NPAD);
        const uint32_t qa = qslot_addr + (uint32_t)slot * kQBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t half = (uint32_t)(kk >> 2), step = (uint32_t)(kk & 3) * 32u;
          const uint64_t ad = sm100::desc_k_sw128(sa + half * (kKeyBytes / 2) + step);
          const uint64_t bd = sm100::desc_k_sw128(qa + half * (kQBytes / 2) + step);
          sm100::mma_bf16(tbuf, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        sm100::mma_commit(&bar_mma[g]);
      }
      issued = true;
      const uint32_t rows = s_trows[s][row];
      // key norm of this thread's row while the MMAs run (the order of the 16-byte granules
      // does not matter): bf16 squares fused into four fp32 sums (exact products, round to
      // nearest). 128 roundings of nonnegative sums stay below 2^-17 relative, so scaling
      // the sum up by 1 + 2^-16 and rounding the root up keeps kn an upper bound of the norm.
      float ka[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const uint8_t* kr = base_ptr + (size_t)s * kKeyBytes + hlf * (kKeyBytes / 2) + row * 128;
#pragma unroll
        for (int gg = 0; gg < 8; ++gg) {
          const uint4 u = *reinterpret_cast<const uint4*>(kr + (((gg + row) & 7) << 4));
          ka[0] = fma2_bf16(u.x, u.x, ka[0]);
          ka[1] = fma2_bf16(u.y, u.y, ka[1]);
          ka[2] = fma2_bf16(u.z, u.z, ka[2]);
          ka[3] = fma2_bf16(u.w, u.w, ka[3]);
        }
      }
      const float kss = __fmul_ru(__fadd_ru(__fadd_ru(ka[0], ka[1]), __fadd_ru(ka[2], ka[3])),
                                  1.0000153f);
      const float kn = __fmul_ru(__fsqrt_ru(kss), 1.0000153f);
      ok = sm100::mbar_wait(&bar_mma[g], mphase, kWaitPolls);
      ok = bar_and(bar_id, 128, ok);
      if (!ok) {
        if (warp == kTcProducerWarps + 4 * g) give_up();
        break;
      }
      issued = false;
      mphase ^= 1u;
      // keys, queries and weights of the stage are read (the MMAs are complete and this
      // thread's key norm is formed): release it before the scores are formed
      __syncwarp();
      if (lane == 0) mbar_arrive1(&bar_empty[s]);
      sm100::tc_fence_after();
      float d[NPAD];
      const uint32_t lane_base = tbuf + ((uint32_t)((warp & 3) * 32) << 16);
#pragma unroll
      for (int c = 0; c < NCH; ++c) sm100::tmem_ld16(lane_base + (uint32_t)(c * 16), d + c * 16);
      sm100::tc_fence_before();   // the group barrier of the next tile orders the next MMA
      const int e = e0 + row;
      // Per row: the score (every lane forms it; keys past the layer's union are zero
      // rows), stored for the entries of the union. Per chunk of 32 entries (this warp's;
      // a tile starts at a multiple of 128 entries): the largest key norm bound kc, which
      // K7's first test takes in place of each entry's own, and per row the largest
      // admitted score (-inf: none), which with kc bounds the chunk's intervals for K7's
      // threshold and first test. The chunk's values leave in one store (lane r < R: row
      // r's maximum, lane R: kc), next to the gather's copies in the memory pipe.
      const bool live = e < ucnt;
      const bool chunk_live = e0 + (warp & 3) * 32 < ucnt;   // warp-uniform
      if (live) st_hint(a.knorm + (size_t)l * a.NS + e, kn, spol);
      auto emit = [&](int r, float sc) {
        const bool adm = live && (rows & (1u << r));
        if (live)
          st_hint(a.sc0 + ((size_t)l * R + r) * a.NS + e,
                  adm ? __float_as_uint(sc) : kMinusInfBits, spol);
        return adm ? sc : -INFINITY;
      };
      const size_t cidx = (size_t)l * a.NC + (e0 >> 5) + (warp & 3);   // the chunk
      if constexpr (HH > 0) {   // head count known at compile time: static indices
        constexpr int NR = NPAD / HH < 8 ? NPAD / HH : 8;
        // values 0 .. R-1: the rows' scores, value R (R < 8): kn; reduced together
        float v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) v[r] = -INFINITY;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (r < R) {
            float sc = 0.0f;
#pragma unroll
            for (int h = 0; h < HH; ++h) {
              const float x = d[r * HH + h];
              sc = __fmaf_rn(s_wg[g][r * HH + h], x > 0.0f ? x : 0.0f, sc);
            }
            v[r] = emit(r, sc);
          }
        }
        const float knv = live ? kn : 0.0f;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r == R) v[r] = knv;
        const float kc8 = R < 8 ? 0.0f : warp_max(knv);
        const float mine = warp_max8(v);
        const int slot = (lane >> 2) & 7;   // the value this lane holds: 4 b4 + 2 b3 + b2
        const int which = (lane & 3) == 0 ? slot : 8;
        if (chunk_live && which < R) st_hint(a.smax + cidx * R + which, mine, spol);
        if (chunk_live && (R < 8 ? which == R : lane == 0))
          st_hint(a.kmax + cidx, R < 8 ? mine : kc8, spol);
      } else {                  // any head count: each row picks its columns by predicate
        float mine = warp_max(live ? kn : 0.0f);   // lane r < R: row r's largest; lane R: kc
#pragma unroll 1
        for (int r = 0; r < R; ++r) {
          const int p0 = r * Hh, p1 = p0 + Hh;
          float sc = 0.0f;
#pragma unroll
          for (int p = 0; p < NPAD; ++p) {
            const float x = d[p];
            const float t = __fmaf_rn(s_wg[g][p], x > 0.0f ? x : 0.0f, sc);
            sc = (p >= p0 && p < p1) ? t : sc;
          }
          const float mx = warp_max(emit(r, sc));
          if (lane == r) mine = mx;
        }
        if (chunk_live && lane <= R) st_hint(lane < R ? a.smax + cidx * R + lane : a.kmax + cidx, mine, spol);
      }
    }
    // MMAs issued but never observed complete: wait (bounded) before TMEM is freed
    if (issued) sm100::mbar_wait(&bar_mma[g], mphase, kWaitPolls);
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, G::kTmemCols);
}

// ---------------------------------------------------------------------------------
// K7 building blocks. Each warp owns a contiguous segment of the row's entries and walks
// it 32 at a time (coalesced loads, several batches in flight); per-warp counts are
// combined once where an ordered result is needed.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void warp_segment(int n, int* beg, int* end) {
  const int warp = threadIdx.x >> 5;
  const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
  *beg = warp * seg;
  *end = min(n, *beg + seg);
}

// One histogram pass of the radix select over digit (key >> shift) & 255 of the elements
// whose higher digits equal `prefix` (all elements when `first`). One shared atomic per
// distinct bucket per warp: scores cluster in a few top-byte buckets.
template <typename KeyAt>
__device__ __forceinline__ void hist_pass(int n, bool resid, const uint32_t* r_key, int rn,
                                          int shift, uint32_t prefix, bool first,
                                          KeyAt key_at, int* hist) {
  const int lane = threadIdx.x & 31;
  auto add = [&](uint32_t key, bool valid) {
    const bool in = valid && (first || (key >> (shift + 8)) == prefix);
    const uint32_t bucket = in ? ((key >> shift) & 255u) : 256u;
    const unsigned peers = __match_any_sync(0xffffffffu, bucket);
    if (in && lane == (__ffs(peers) - 1)) atomicAdd(&hist[bucket], __popc(peers));
  };
  if (resid) {
    for (int i0 = 0; i0 < rn; i0 += blockDim.x) {
      const int i = i0 + threadIdx.x;
      add(i < rn ? r_key[i] : 0u, i < rn);
    }
  } else {
    constexpr int U = 8;
    int beg, end;
    warp_segment(n, &beg, &end);
    for (int i0 = beg; i0 < end; i0 += 32 * U) {
      uint32_t k[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * 32 + lane;
        k[u] = i < end ? key_at(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)   // (warp-uniform) groups past the segment are skipped
        if (i0 + u * 32 < end) add(k[u], i0 + u * 32 + lane < end);
    }
  }
}

// The key of the need-th largest element among n keys, MSB-first 8 bits at a time. After
// the first two passes the elements whose top 16 bits match are gathered into r_key (if
// at most kResidCap of them) and the last two passes run there. Two block barriers per
// pass: one after the histogram (hist holds two 256-bin buffers, the next pass's cleared
// while this one fills), one after warp 0 has found the bucket (8 bins per lane, a warp
// scan). *need_out = how many elements equal to the threshold belong to the selection.
// All threads must call it.
// With start > 0 the first `start` digits are given (prefix0): every element that can
// reach the threshold has them, and the elements that do not are counted below it.
template <typename KeyAt>
__device__ uint32_t radix_threshold(int n, int need, KeyAt key_at, int* hist, int* scratch,
                                    uint32_t* r_key, int* s_misc, uint32_t* status,
                                    int* need_out, int passes = 4, int start = 0,
                                    uint32_t prefix0 = 0u) {
  (void)scratch;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int& s_bucket = s_misc[0];
  int& s_need = s_misc[1];
  int& s_rn = s_misc[2];
  int& s_cnt = s_misc[3];   // elements in the chosen bucket
  uint32_t prefix = prefix0;
  bool resid = false;
  for (int i = tid; i < 256; i += blockDim.x) hist[(start & 1) * 256 + i] = 0;
  __syncthreads();
  for (int pass = start; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    int* h = hist + (pass & 1) * 256;
    if (tid == 0 && pass == 1) s_rn = 0;
    hist_pass(n, resid, r_key, resid ? min(s_rn, kResidCap) : 0, shift, prefix,
              pass == 0, key_at, h);
    for (int i = tid; i < 256; i += blockDim.x) hist[((pass + 1) & 1) * 256 + i] = 0;
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8l down to 248 - 8l (descending keys)
      int v[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[q] = h[255 - 8 * lane - q];
        sum += v[q];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int acc = incl - sum, bucket = -1, nneed = need, bcnt = 0;
      if (acc < need && need <= incl) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (bucket < 0 && acc < need && need <= acc + v[q]) {
            bucket = 255 - 8 * lane - q;
            nneed = need - acc;
            bcnt = v[q];
          }
          acc += v[q];
        }
      }
      const unsigned found = __ballot_sync(0xffffffffu, bucket >= 0);
      if (bucket >= 0) {
        s_bucket = bucket;
        s_need = nneed;
        s_cnt = bcnt;
      }
      if (!found && lane == 0) {   // histogram inconsistent with `need`: report
        flag_status(status, kStatusCheck);
        s_bucket = 0;
        s_need = need;
        s_cnt = h[255];
      }
    }
    __syncthreads();
    const int b = s_bucket;
    const int cnt = s_cnt;   // (h may be cleared by a thread already in the next pass)
    prefix = (prefix << 8) | (uint32_t)b;
    need = s_need;
    if (pass == 1 && !resid && passes > 2) {
      if (cnt <= kResidCap) {
        constexpr int U = 8;
        int beg, end;
        warp_segment(n, &beg, &end);
        for (int i0 = beg; i0 < end; i0 += 32 * U) {
          uint32_t k[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = i0 + u * 32 + lane;
            k[u] = i < end ? key_at(i) : 0u;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int i = i0 + u * 32 + lane;
            if (i < end && (k[u] >> 16) == prefix) {
              const int p = atomicAdd(&s_rn, 1);
              if (p < kResidCap) r_key[p] = k[u];
            }
          }
        }
        __syncthreads();
        resid = true;
        if (s_rn != cnt && tid == 0) flag_status(status, kStatusCheck);
      }
    }
  }
  __syncthreads();   // s_misc and hist are free for the caller
  *need_out = need;
  return prefix << (32 - 8 * passes);   // with fewer passes: the bucket's lower bound
}

// Ordered selection over n elements: every element classified 2 ("greater"), plus the
// first `need` elements (in index order) classified 1 ("equal"); emit(pos, i) for each,
// pos ascending from 0. Two passes over the warps' segments with the per-warp counts
// combined in between. Returns how many were taken. All threads must call it.
template <typename Cls, typename Emit>
__device__ int ordered_take(int n, int need, Cls cls, Emit emit, int* s_eq, int* s_gt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int beg, end;
  warp_segment(n, &beg, &end);
  constexpr int U = 8;
  int gt_w = 0, eq_w = 0;
  for (int i0 = beg; i0 < end; i0 += 32 * U) {
    int c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * 32 + lane;
      c[u] = i < end ? cls(i) : 0;        // 2 = greater, 1 = equal, 0 = below
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {   // (warp-uniform) groups past the segment are skipped
      if (i0 + u * 32 >= end) break;
      gt_w += __popc(__ballot_sync(0xffffffffu, c[u] == 2));
      eq_w += __popc(__ballot_sync(0xffffffffu, c[u] == 1));
    }
  }
  if (lane == 0) { s_eq[warp] = eq_w; s_gt[warp] = gt_w; }
  __syncthreads();
  int eq_acc = 0, out_acc = 0, my_eq = 0, my_out = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    if (w == warp) { my_eq = eq_acc; my_out = out_acc; }
    out_acc += s_gt[w] + max(0, min(s_eq[w], need - eq_acc));
    eq_acc += s_eq[w];
  }
  int pos = my_out, eq_seen = my_eq;
  for (int i0 = beg; i0 < end; i0 += 32 * U) {
    int c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * 32 + lane;
      c[u] = i < end ? cls(i) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i0 + u * 32 >= end) break;
      const int i = i0 + u * 32 + lane;
      const uint32_t eqm = __ballot_sync(0xffffffffu, c[u] == 1);
      const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
      const bool take = (c[u] == 2) || (c[u] == 1 && eq_rank < need);
      const uint32_t tm = __ballot_sync(0xffffffffu, take);
      if (take) emit(pos + __popc(tm & ((1u << lane) - 1u)), i);
      pos += __popc(tm);
      eq_seen += __popc(eqm);
    }
  }
  __syncthreads();
  return out_acc;
}

// ---------------------------------------------------------------------------------
// K7: bounded radix top-k, one CTA of 512 threads per (layer, row), over the layer's union
// entries (entries the row does not admit carry the sentinel and never qualify).
// Canonical mode: threshold and ordered take over the canonical scores.
// Tensor-core mode, all inside the CTA:
//  1. tau, a collection threshold at or below the K-th largest lower bound: the K-th largest
//     of the per-chunk bounds RD(smax - RU(kc G)) (each reached by a lower bound in its
//     chunk), to two digits (the bucket's lower bound); when fewer than K chunks hold an
//     admitted entry, from a sample of 2048 entries (64 chunks of 32, evenly spaced) at
//     rank K scaled to the sample plus 16. Rows that fit the collection whole take tau = 0.
//  2. collection: the entries whose upper bound reaches tau, in index order, with their
//     bounds and block ids, and how many of them have a lower bound >= tau. Each warp walks
//     a contiguous segment in two passes (the scores alone against a threshold per 32
//     entries, in the chunks whose largest score reaches it; then the exact bounds of the
//     entries that pass) and keeps its matches in
//     shared memory; the warps' lists are concatenated.
//  3. If at least K lower bounds reach tau, the K-th largest lower bound T of the row is
//     among the collected entries and so is every candidate (upper bound >= T). Otherwise
//     (or on overflow) T and the candidates come from two passes over the whole row.
//  4. Candidates whose lower bound exceeds H (below) are selected whatever the exact scores;
//     the others are re-scored in the canonical order.
//  5. The exact select among the candidates, ties to the lowest index: the uncertain ones
//     sorted by (key, position) when at most one per thread remains, else a threshold over
//     all candidates' keys (the certain ones carry the largest key); the ordered take.
// With more candidates than the CTA keeps: canonical re-score of every admitted entry of
// the row, then the canonical-mode path. At the end the row's scores (and, after the
// layer's last row, the layer's key norms and union lists) are dropped from L2.
// ---------------------------------------------------------------------------------
struct TopkArgs {
  int R, Hh, N, K;
  int64_t key_stride;
  const uint16_t* keys;
  const uint16_t* q;
  const float* hw;
  const int32_t* cidx;
  const int32_t* ccount;
  const int32_t* uidx;
  const int32_t* ucount;
  uint32_t* sc0;
  const float* knorm;
  const float* qnorm;
  const float* kmax;
  int32_t* sel;
  int32_t* nsel;
  uint32_t* status;
  int tc_mode;
  int NS;             // row stride of sc0 / knorm (N rounded up to a multiple of 32)
  int NC;             // row stride of kmax
  uint32_t* ldone;    // [L] rows done per layer
  const uint8_t* urows;
  int keep;           // leave the scores, key norms and union lists in the workspace
  const float* smax;  // [L][NC][R] per 32 union entries, each row's largest score
                      // (-inf: none admitted; tensor-core mode)
};

// Drops the 128-byte lines that lie wholly inside [p, p + bytes) from L2 without writing
// them back (their contents become undefined), spread over the block's threads.
__device__ __forceinline__ void discard_lines(const void* p, size_t bytes) {
  const uintptr_t a0 = (reinterpret_cast<uintptr_t>(p) + 127) & ~(uintptr_t)127;
  const uintptr_t a1 = (reinterpret_cast<uintptr_t>(p) + bytes) & ~(uintptr_t)127;
  for (uintptr_t x = a0 + 128 * threadIdx.x; x < a1; x += 128 * (uintptr_t)blockDim.x)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(x) : "memory");
}

// Bitonic sort, descending, of one 64-bit value per thread over threads 0 .. P - 1 (P a
// power of two <= the block size; the other threads sort their own values among
// themselves): returns the value of this thread's rank. Exchanges within a warp go by
// shuffles, wider ones through buf (2 x blockDim.x values, alternating, one barrier each).
// All threads must call it.
__device__ uint64_t block_sort_desc(uint64_t v, int P, uint64_t* buf) {
  const int tid = threadIdx.x;
  int step = 0;
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      uint64_t o;
      if (j >= 32) {
        uint64_t* b = buf + (step & 1) * blockDim.x;
        b[tid] = v;
        __syncthreads();
        o = b[tid ^ j];
        ++step;
      } else {
        o = __shfl_xor_sync(0xffffffffu, v, j);
      }
      const bool lower = (tid & j) == 0, first_half_up = (tid & k) == 0;
      v = (lower == first_half_up) ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

constexpr int kWarpBuf = 256;   // collected entries a warp keeps before the lists merge
constexpr int kRescoreRound = 96;    // uncertain candidates re-scored per round (<= threads / 4)
constexpr int kRescoreBuf = kRescoreRound * 256;   // one round's staged keys (two alternate)
// dynamic shared memory of K7: residual keys, candidates and their keys, the row's queries
// (fp32, [i][head]) and head weights, the collection (block id, lower and upper bound key),
// the queries again as bf16 pairs for up to 8 heads
constexpr size_t kTopkSmem = sizeof(uint32_t) * kResidCap + sizeof(int32_t) * 2 * kCandCap +
                             sizeof(float) * (kScoreMaxHeads * 128 + kScoreMaxHeads) +
                             sizeof(int32_t) * 3 * kCollectCap + sizeof(uint32_t) * 4 * 128;
// the warps' collection lists live over the residual keys and the candidates
static_assert((size_t)3 * kTopkWarps * kWarpBuf <= (size_t)kResidCap + 2 * kCandCap,
              "collection lists overlap the queries");
static_assert(kCollectCap >= 2048, "the tau sample lives over the collection");
static_assert((size_t)2 * kRescoreBuf <= sizeof(int32_t) * 3 * kCollectCap,
              "key staging overlaps past the collection");
static_assert(4 * kRescoreRound <= kTopkThreads, "four threads per candidate");
static_assert(kScoreMaxHeads == 16, "four threads of four heads each per candidate");

__global__ void __launch_bounds__(kTopkThreads, 2) k7_topk(TopkArgs a) {
  __shared__ int hist[512];   // two radix histogram buffers
  __shared__ int scratch[33];
  __shared__ int s_misc[4];
  __shared__ int s_eq[kTopkWarps], s_gt[kTopkWarps];
  __shared__ int s_cnt[kTopkWarps], s_lo[kTopkWarps];
  __shared__ unsigned s_dmax, s_maxlo;
  extern __shared__ __align__(16) uint8_t dsm[];
  uint32_t* r_key = reinterpret_cast<uint32_t*>(dsm);              // [kResidCap]
  int32_t* cand = reinterpret_cast<int32_t*>(r_key + kResidCap);   // [kCandCap]
  uint32_t* ckey = reinterpret_cast<uint32_t*>(cand + kCandCap);   // [kCandCap]
  float* qf = reinterpret_cast<float*>(ckey + kCandCap);           // [128][kScoreMaxHeads]
  float* wf = qf + kScoreMaxHeads * 128;                           // [Hh]
  int32_t* col_i = reinterpret_cast<int32_t*>(wf + kScoreMaxHeads);
  uint32_t* col_lo = reinterpret_cast<uint32_t*>(col_i + kCollectCap);
  uint32_t* col_hi = col_lo + kCollectCap;
  // [i / 4][t][i % 4]: bf16 pair (head t, head t + 4) of query value i, t = 0..3
  uint32_t* qb = col_hi + kCollectCap;
  uint32_t* const wbuf = r_key;                                    // [warp][3][kWarpBuf]
  uint32_t* const samp = reinterpret_cast<uint32_t*>(col_i);       // [2048]

  // the row's queries as fp32 in the [i][head] layout (heads at qslot(h), heads past Hh
  // zero) and its head weights
  auto stage_queries = [&]() {
    const int tid = threadIdx.x;
    for (int i = tid; i < a.Hh; i += blockDim.x) wf[i] = a.hw[(size_t)blockIdx.x * a.Hh + i];
    for (int i = a.Hh * 128 + tid; i < kScoreMaxHeads * 128; i += blockDim.x)
      qf[(i & 127) * kScoreMaxHeads + qslot(i >> 7)] = 0.0f;
    const uint16_t* qrow = a.q + (size_t)blockIdx.x * a.Hh * 128;
    for (int i = tid; i < a.Hh * 128; i += blockDim.x)
      qf[(i & 127) * kScoreMaxHeads + qslot(i >> 7)] = bf16_bits_to_f32(qrow[i]);
    if (a.Hh <= 8) {
      for (int w = tid; w < 4 * 128; w += blockDim.x) {
        const int i = w & 127, t = w >> 7;   // value i of heads t (low half) and t + 4
        const uint32_t lo = t < a.Hh ? qrow[t * 128 + i] : 0u;
        const uint32_t hi = t + 4 < a.Hh ? qrow[(t + 4) * 128 + i] : 0u;
        qb[((i >> 2) * 4 + t) * 4 + (i & 3)] = lo | (hi << 16);
      }
    }
  };

  // The queries are inputs of the call: staged (for the re-scores of tensor-core mode)
  // while the scoring grid finishes.
  if (a.tc_mode) stage_queries();
  pdl_wait();   // the scores and the compaction are complete
  pdl_trigger();
  if (threadIdx.x == 0) s_maxlo = 0u;
  const int lr = blockIdx.x;
  const int l = lr / a.R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the row's admitted count, the layer's union count and the row's interval scale, loaded
  // together
  const int count = a.ccount[lr];
  const int n = a.ucount[l];
  const float G = a.tc_mode ? a.qnorm[lr] : 0.0f;   // eps per unit key norm
  const int K = a.K;
  int32_t* out = a.sel + (size_t)lr * K;
  // At the end of the row: its scores are dead, and once the layer's last row is done, so
  // are the layer's key norms and union lists. They are dropped from L2 rather than left
  // dirty there (the next kernels would pay for writing them back), unless the caller keeps
  // the workspace for inspection.
  auto finish = [&]() {
    if (a.keep) return;
    __syncthreads();   // every read of this row's data is done
    discard_lines(a.sc0 + (size_t)lr * a.NS, sizeof(uint32_t) * (size_t)a.NS);
    if (tid == 0) s_misc[0] = atomicAdd(a.ldone + l, 1u) == (uint32_t)(a.R - 1) ? 1 : 0;
    __syncthreads();
    if (s_misc[0]) {
      discard_lines(a.knorm + (size_t)l * a.NS, sizeof(float) * (size_t)a.NS);
      if (a.tc_mode) discard_lines(a.smax + (size_t)l * a.NC * a.R, sizeof(float) * a.NC * a.R);
      discard_lines(a.uidx + (size_t)l * a.N, sizeof(int32_t) * (size_t)a.N);
      discard_lines(a.urows + (size_t)l * a.N, (size_t)a.N);
    }
  };

  if (count <= K) {
    const int32_t* ci = a.cidx + (size_t)lr * a.N;
    for (int i = tid; i < K; i += blockDim.x) out[i] = i < count ? ci[i] : -1;
    if (tid == 0) a.nsel[lr] = count;
    finish();
    return;
  }

  const int32_t* ui = a.uidx + (size_t)l * a.N;
  uint32_t* s0 = a.sc0 + (size_t)lr * a.NS;
  const uint16_t* kbase = a.keys + (size_t)l * a.key_stride;
  bool canonical = !a.tc_mode;
  if (a.tc_mode) {
    const float* kn = a.knorm + (size_t)l * a.NS;
    // ---- 1. tau: a key that (at least, or very likely) K lower bounds of the row reach.
    // Each chunk of 32 entries carries its largest score smax (K5) and largest key norm
    // bound kc, so the entry holding smax has a lower bound of at least
    // v = RD(smax - RU(kc G)) (its own kn is at most kc). At least K chunks, each through
    // one of its entries, reach the K-th largest v, so that value, or a lower one (its
    // first two radix digits), is a tau. When fewer than K chunks hold an admitted entry
    // it is zero; a sample of the entries' lower bounds then estimates one (rank a little
    // above K; the collection checks the count).
    uint32_t tau = 0u;
    const int nc = (n + 31) >> 5;
    const float* kc_row = a.kmax + (size_t)l * a.NC;
    // smax of chunk c for this row: sm_row[c * R]
    const uint32_t* sm_row =
        reinterpret_cast<const uint32_t*>(a.smax) + (size_t)l * a.NC * a.R + (lr - l * a.R);
    if (n > kCollectCap && nc >= K) {
      int need;
      if (nc <= kCollectCap) {
        constexpr int kPer = kCollectCap / kTopkThreads;
        uint32_t sv[kPer];
        float kv[kPer];
#pragma unroll
        for (int t = 0; t < kPer; ++t) {   // every load in flight, then the stores
          const int c = tid + t * kTopkThreads;
          sv[t] = c < nc ? sm_row[(size_t)c * a.R] : kMinusInfBits;
          kv[t] = c < nc ? kc_row[c] : 0.0f;
        }
#pragma unroll
        for (int t = 0; t < kPer; ++t) samp[tid + t * kTopkThreads] = tc_lo(sv[t], kv[t], G);
        __syncthreads();
        tau = radix_threshold(nc, K, [&](int c) { return samp[c]; }, hist, scratch, nullptr,
                              s_misc, a.status, &need, 2);
      } else {
        tau = radix_threshold(nc, K, [&](int c) { return tc_lo(sm_row[(size_t)c * a.R], kc_row[c], G); },
                              hist, scratch, nullptr, s_misc, a.status, &need, 2);
      }
    }
    if (n > kCollectCap && tau == 0u) {
      constexpr int kChunks = 64, kS = kChunks * 32;
      const int spacing = n / kChunks;
      static_assert(kS % kTopkThreads == 0, "whole sample rounds");
      constexpr int kPer = kS / kTopkThreads;
      uint32_t sb[kPer];
      float kb[kPer];
#pragma unroll
      for (int t = 0; t < kPer; ++t) {   // every load in flight, then the stores
        const int j = tid + t * kTopkThreads;
        const int i = (j >> 5) * spacing + (j & 31);
        sb[t] = s0[i];
        kb[t] = kn[i];
      }
#pragma unroll
      for (int t = 0; t < kPer; ++t) samp[tid + t * kTopkThreads] = tc_lo(sb[t], kb[t], G);
      __syncthreads();
      const int rank = min(kS, (int)(((long long)K * kS + n - 1) / n) + 16);
      int need;
      tau = radix_threshold(kS, rank, [&](int j) { return samp[j]; }, hist, scratch, nullptr,
                            s_misc, a.status, &need, 2);
    }
    // ---- 2. collection, in two passes per warp. Each warp walks a contiguous segment
    // (starting at a multiple of 128 entries); entries past `end` in the last group lie
    // inside the row's padded stride and are masked.
    //   Pass 1 reads only the chunks' largest upper bounds and, in the chunks where one
    // reaches tau, the scores: 16 consecutive entries per lane, and keeps those with
    // s >= theta,
    // theta = RD(RD(t* - A) - RU(2^-22 |t*| + 2^-126)), A = RU(kc G), where kc >= kn is the
    // largest key norm bound of the entry's 32 and t* the smallest score whose key reaches
    // tau. This keeps every entry the exact test takes: if RU(z) >= t* for
    // z = s + RU(kn G), then z >= t* - ulp(z) >= t* - 2^-22 |t*| - 2^-149, and
    // RU(kn G) <= A, so s >= t* - A - 2^-22 |t*| - 2^-149 >= theta. An entry the row does
    // not admit (s = -inf) never passes; tau at or below the key of -inf takes every
    // entry. The passing entries' positions are listed in order (a lane's place is the
    // prefix over the lanes of their counts, by bit-sliced ballots).
    //   Pass 2 takes the listed entries 32 at a time (all loads of a lane issued first),
    // forms their exact bounds from the entry's own kn and keeps, in order and in place,
    // the ones whose upper bound reaches tau, with their block ids and both bounds,
    // counting the lower bounds that reach tau.
    int m = -1;
    __syncthreads();   // s_maxlo is zero
    {
      const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 127) & ~127;
      const int beg = min(n, warp * seg), end = min(n, beg + seg);
      uint32_t* const b_i = wbuf + (size_t)warp * 3 * kWarpBuf;
      uint32_t* const b_lo = b_i + kWarpBuf;
      uint32_t* const b_hi = b_lo + kWarpBuf;
      const bool take_all = tau <= 0x007FFFFFu;
      const float tstar = key_score(tau);
      const unsigned lt = (1u << lane) - 1u;
      int c1 = 0;   // entries that pass the first test (listed while c1 < kWarpBuf)
      {
        const uint64_t rpol = l2_evict_first_policy();   // each score is read once here
        // the first test's margin (see above), formed rounding upward
        const float mt = __fmaf_ru(0.0000002384185791015625f, fabsf(tstar), 1.17549435e-38f);
        const uint32_t all16 = take_all ? 0xFFFFu : 0u;
        const uint4 kNone = make_uint4(kMinusInfBits, kMinusInfBits, kMinusInfBits, kMinusInfBits);
        // The chunks of 32 entries (one kc each) where an entry passes, i.e. whose largest
        // score reaches theta (all of them when every entry is taken), are listed in order,
        // 32 chunks at a time (the next 32 chunks' smax and kc in flight); lane L then takes
        // half L & 1 (16 consecutive entries, four 16-byte loads) of listed chunk L >> 1,
        // 16 listed chunks per batch.
        uint32_t* const clist = b_lo;   // free until the second pass
        const int cbeg = beg >> 5, cend = beg < end ? (end + 31) >> 5 : cbeg;   // none: empty
        float hs = cbeg + lane < cend ? __uint_as_float(sm_row[(size_t)(cbeg + lane) * a.R]) : -INFINITY;
        float hk = cbeg + lane < cend ? kc_row[cbeg + lane] : 0.0f;
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          const int c = c0 + lane;
          const bool cp = c < cend &&
                          (take_all || hs >= __fsub_rd(__fsub_rd(tstar, __fmul_ru(hk, G)), mt));
          if (c0 + 32 < cend) {
            hs = c + 32 < cend ? __uint_as_float(sm_row[(size_t)(c + 32) * a.R]) : -INFINITY;
            hk = c + 32 < cend ? kc_row[c + 32] : 0.0f;
          }
          const unsigned M = __ballot_sync(0xffffffffu, cp);
          if (cp) clist[__popc(M & lt)] = (uint32_t)c;
          __syncwarp();
          const int np = __popc(M);
          for (int j0 = 0; j0 < np; j0 += 16) {
            const int j = j0 + (lane >> 1);
            const int cc = j < np ? (int)clist[j] : -1;
            const int i = cc * 32 + 16 * (lane & 1);
            const int lim = cc < 0 ? 0 : end - i;   // entries of this lane inside the segment
            uint4 sv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) sv[q] = 4 * q < lim ? ld_hint_v4(s0 + i + 4 * q, rpol) : kNone;
            const float kc = cc >= 0 ? kc_row[cc] : 0.0f;
            const float th = __fsub_rd(__fsub_rd(tstar, __fmul_ru(kc, G)), mt);
            uint32_t pm = all16;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              pm |= __uint_as_float(sv[q].x) >= th ? 1u << (4 * q) : 0u;
              pm |= __uint_as_float(sv[q].y) >= th ? 2u << (4 * q) : 0u;
              pm |= __uint_as_float(sv[q].z) >= th ? 4u << (4 * q) : 0u;
              pm |= __uint_as_float(sv[q].w) >= th ? 8u << (4 * q) : 0u;
            }
            pm &= lim >= 16 ? 0xFFFFu : (lim > 0 ? (1u << lim) - 1u : 0u);
            if (__ballot_sync(0xffffffffu, pm != 0u)) {
              const int cn = __popc(pm);   // 0..16: five bit slices
              int p = c1, tot = 0;
#pragma unroll
              for (int bit = 0; bit < 5; ++bit) {
                const unsigned sl = __ballot_sync(0xffffffffu, (cn >> bit) & 1);
                p += __popc(sl & lt) << bit;
                tot += __popc(sl) << bit;
              }
              while (pm) {
                const int e = __ffs(pm) - 1;
                pm &= pm - 1u;
                if (p < kWarpBuf) b_i[p] = (uint32_t)(i + e);
                ++p;
              }
              c1 += tot;
            }
          }
          __syncwarp();   // the list is rewritten by the next step
        }
      }
      __syncwarp();
      int cnt = 0, nlo = 0;
      if (c1 > kWarpBuf) {
        cnt = c1;   // the list overflowed: the slow path below
      } else {
        constexpr int P = kWarpBuf / 32;
        uint32_t ii[P], sb[P];
        float kk[P];
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const int p = 32 * j + lane;
          const uint32_t e = p < c1 ? b_i[p] : 0u;
          sb[j] = p < c1 ? s0[e] : kMinusInfBits;
          kk[j] = p < c1 ? kn[e] : 0.0f;
          ii[j] = p < c1 ? (uint32_t)ui[e] : 0u;   // the entry's block id
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < P; ++j) {
          if (32 * j >= c1) break;
          const bool valid = 32 * j + lane < c1;
          const uint32_t hk = valid ? tc_hi(sb[j], kk[j], G) : 0u;
          const bool take = valid && hk >= tau;
          const unsigned bal = __ballot_sync(0xffffffffu, take);
          if (take) {
            const uint32_t lk = tc_lo(sb[j], kk[j], G);
            const int w = cnt + __popc(bal & lt);
            b_i[w] = ii[j];
            b_lo[w] = lk;
            b_hi[w] = hk;
            nlo += lk >= tau ? 1 : 0;
          }
          cnt += __popc(bal);
        }
        // the largest lower bound collected
        __syncwarp();
        uint32_t ml = 0u;
        for (int p = lane; p < cnt; p += 32) ml = max(ml, b_lo[p]);
        ml = __reduce_max_sync(0xffffffffu, ml);
        if (lane == 0 && ml) atomicMax(&s_maxlo, ml);
      }
      nlo = __reduce_add_sync(0xffffffffu, nlo);
      if (lane == 0) { s_cnt[warp] = cnt; s_lo[warp] = nlo; }
      __syncthreads();
      int off = 0, total = 0, lo_total = 0;
      bool over = false;
      for (int w = 0; w < kTopkWarps; ++w) {
        if (w == warp) off = total;
        total += s_cnt[w];
        lo_total += s_lo[w];
        over |= s_cnt[w] > kWarpBuf;
      }
      const bool fast = !over && total <= kCollectCap && lo_total >= K;
      if (fast)
        for (int p = lane; p < cnt; p += 32) {
          col_i[off + p] = b_i[p];   // the entry's block id
          col_lo[off + p] = b_lo[p];
          col_hi[off + p] = b_hi[p];
        }
      __syncthreads();
      // ---- 3./4. over the collection: T, the candidates and the certain ones
      if (fast) {
        // At least K lower bounds reach tau, so T >= tau, and every lower bound at or
        // above tau shares the leading bytes of tau and of the largest lower bound: those
        // digits are given.
        const uint32_t dx = tau ^ s_maxlo;
        const int start = min(3, dx == 0u ? 4 : __clz((int)dx) >> 3);
        int need;
        const uint32_t T = radix_threshold(
            total, K, [&](int j) { return col_lo[j]; }, hist, scratch, r_key, s_misc, a.status,
            &need, 4, start, start > 0 ? tau >> (32 - 8 * start) : 0u);
        // H = T + max over the candidates of (upper - lower), rounded upward, is at least
        // the (K+1)-th largest upper bound of the row (the K+1 largest upper bounds each
        // exceed their lower bound by at most that much, and at most K lower bounds reach
        // past T). A candidate whose lower bound exceeds H is beaten by fewer than K others
        // whatever the exact scores: it is selected without being re-scored, and takes the
        // key kCertainKey so that the exact select below keeps it.
        if (tid == 0) s_dmax = 0u;
        __syncthreads();
        {
          float dm = 0.0f;
          for (int j = tid; j < total; j += blockDim.x)
            if (col_hi[j] >= T)
              dm = fmaxf(dm, __fsub_ru(key_score(col_hi[j]), key_score(col_lo[j])));
          dm = warp_max(dm);
          if (lane == 0) atomicMax(&s_dmax, __float_as_uint(dm));   // dm >= 0
        }
        __syncthreads();
        const uint32_t Hk = score_key(__fadd_ru(key_score(T), __uint_as_float(s_dmax)));
        m = ordered_take(
            total, 0, [&](int j) { return col_hi[j] >= T ? 2 : 0; },
            [&](int p, int j) {
              if (p < kCandCap) {
                cand[p] = col_i[j];
                ckey[p] = col_lo[j] > Hk ? kCertainKey : 0u;
              }
            },
            s_eq, s_gt);
      }
    }
    bool cand_entries = false;   // cand holds union entries (else block ids)
    if (m < 0) {
      // exact T over the whole row, then the ordered gather of the candidates (upper bound
      // reaches T), bounded by kCandCap; none is taken as certain
      cand_entries = true;
      int need;
      const uint32_t T = radix_threshold(
          n, K, [&](int i) { return tc_lo(s0[i], kn[i], G); }, hist, scratch, r_key, s_misc,
          a.status, &need);
      m = ordered_take(
          n, 0, [&](int i) { return tc_hi(s0[i], kn[i], G) >= T ? 2 : 0; },
          [&](int p, int i) {
            if (p < kCandCap) {
              cand[p] = i;
              ckey[p] = 0u;
            }
          },
          s_eq, s_gt);
    }
    __syncthreads();
    if (m <= kCandCap) {
      if (cand_entries)
        for (int j = tid; j < m; j += blockDim.x) cand[j] = ui[cand[j]];
      __syncthreads();
      // ---- 4. canonical scores of the uncertain candidates. Their positions are listed
      // (over the residual keys); rounds of 96 stage their keys in shared memory (two
      // alternating buffers over the collection), and four threads take a candidate: thread t runs
      // the chains of heads t, t + 4, t + 8, t + 12 over i ascending (a fused multiply-add
      // per step), and the first of the four sums the heads' ReLU terms in head order.
      int32_t* const ulist = reinterpret_cast<int32_t*>(r_key);
      int mu = 0;
      {
        if (tid == 0) s_misc[0] = 0;
        __syncthreads();
        for (int j0 = 0; j0 < m; j0 += blockDim.x) {
          const int j = j0 + tid;
          const bool u = j < m && ckey[j] != kCertainKey;
          const unsigned bal = __ballot_sync(0xffffffffu, u);
          int wb = 0;
          if (lane == 0 && bal) wb = atomicAdd(&s_misc[0], __popc(bal));
          wb = __shfl_sync(0xffffffffu, wb, 0);
          if (u) {
            ulist[wb + __popc(bal & ((1u << lane) - 1u))] = j;
            // its key to L2 now: the rounds below copy it from there
            const uint8_t* kp = reinterpret_cast<const uint8_t*>(kbase) + (size_t)cand[j] * 256;
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(kp));
            asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(kp + 128));
          }
        }
        __syncthreads();
        mu = s_misc[0];
        uint8_t* const stg = reinterpret_cast<uint8_t*>(col_i);
        const uint32_t stg_addr = static_cast<uint32_t>(__cvta_generic_to_shared(stg));
        const uint8_t* kb8 = reinterpret_cast<const uint8_t*>(kbase);
        const int sub = tid & 3, slot = tid >> 2;
        const int rounds = (mu + kRescoreRound - 1) / kRescoreRound;
        // round r's keys go to buffer r & 1 (rows of 256 bytes, 16-byte granule c of row
        // j at c ^ (j & 15)); the next round's copies are in flight while this one is
        // scored
        auto stage = [&](int r) {
          const int u0 = r * kRescoreRound, nr = min(kRescoreRound, mu - u0);
          const uint32_t dst = stg_addr + (uint32_t)((r & 1) * kRescoreBuf);
          for (int t = tid; t < nr * 16; t += blockDim.x) {
            const int j = t >> 4, c = t & 15;
            cp_async16(dst + (uint32_t)(j * 256 + ((c ^ (j & 15)) << 4)),
                       kb8 + (size_t)cand[ulist[u0 + j]] * 256 + c * 16, true);
          }
          cp_async_commit();
        };
        if (rounds > 0) stage(0);
        for (int r = 0; r < rounds; ++r) {
          if (r + 1 < rounds) stage(r + 1);
          else cp_async_commit();   // an empty group: the wait below keeps one group open
          cp_async_wait<1>();
          __syncthreads();          // round r's keys are in shared memory
          const int u0 = r * kRescoreRound, nr = min(kRescoreRound, mu - u0);
          const uint8_t* kr = stg + (r & 1) * kRescoreBuf + slot * 256;
          const int sw = slot & 15;
          float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if (slot < nr && a.Hh <= 8) {
            // heads t + 8, t + 12 are absent: two chains per thread on bf16 operands
            const uint32_t* qt = qb + sub * 4;
#pragma unroll 2
            for (int c = 0; c < 16; ++c) {
              const uint4 kv = *reinterpret_cast<const uint4*>(kr + ((c ^ sw) << 4));
              const uint4 q0 = *reinterpret_cast<const uint4*>(qt + (2 * c) * 16);
              const uint4 q1 = *reinterpret_cast<const uint4*>(qt + (2 * c + 1) * 16);
              fma_pair_bf16<false>(d[0], d[1], q0.x, kv.x);
              fma_pair_bf16<true>(d[0], d[1], q0.y, kv.x);
              fma_pair_bf16<false>(d[0], d[1], q0.z, kv.y);
              fma_pair_bf16<true>(d[0], d[1], q0.w, kv.y);
              fma_pair_bf16<false>(d[0], d[1], q1.x, kv.z);
              fma_pair_bf16<true>(d[0], d[1], q1.y, kv.z);
              fma_pair_bf16<false>(d[0], d[1], q1.z, kv.w);
              fma_pair_bf16<true>(d[0], d[1], q1.w, kv.w);
            }
          } else if (slot < nr) {
#pragma unroll 2
            for (int c = 0; c < 16; ++c) {
              const uint4 kv = *reinterpret_cast<const uint4*>(kr + ((c ^ sw) << 4));
              const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                                   bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 qv =
                    *reinterpret_cast<const float4*>(qf + (c * 8 + e) * kScoreMaxHeads + sub * 4);
                d[0] = __fmaf_rn(qv.x, kf[e], d[0]);
                d[1] = __fmaf_rn(qv.y, kf[e], d[1]);
                d[2] = __fmaf_rn(qv.z, kf[e], d[2]);
                d[3] = __fmaf_rn(qv.w, kf[e], d[3]);
              }
            }
          }
          float dh[kScoreMaxHeads];   // head h = 4j + t: d[j] of thread t
#pragma unroll
          for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dh[4 * j + t] = __shfl_sync(0xffffffffu, d[j], (lane & ~3) + t);
          if (sub == 0 && slot < nr) {
            float sc = 0.0f;
#pragma unroll
            for (int h = 0; h < kScoreMaxHeads; ++h)
              if (h < a.Hh) sc = __fmaf_rn(wf[h], dh[h] > 0.0f ? dh[h] : 0.0f, sc);
            ckey[ulist[u0 + slot]] = score_key(sc);
          }
          __syncthreads();   // buffer r & 1 is free for round r + 2
        }
        cp_async_wait<0>();
      }
      // ---- 5. the exact select among the candidates: the first K by (key desc,
      // position asc). The certain ones all belong to it. When at most one uncertain
      // candidate per thread remains (none with the certain key), the uncertain ones are
      // sorted by (key desc, position asc) and the first K - (m - mu) take the certain
      // key; otherwise a radix threshold over all candidates.
      const int need_u = K - (m - mu);
      if (tid == 0) s_misc[1] = 0;
      __syncthreads();
      uint32_t myk = 0u;
      int myj = -1;
      if (tid < mu && mu <= kTopkThreads) {
        myj = ulist[tid];
        myk = ckey[myj];
        if (myk == kCertainKey) s_misc[1] = 1;
      }
      __syncthreads();
      const bool direct = mu <= kTopkThreads && need_u >= 0 && need_u <= mu && !s_misc[1];
      int taken;
      if (direct) {
        if (mu > 0) {
          int P = 2;
          while (P < mu) P <<= 1;
          // (key, complement of the position): descending order is (key desc, position
          // asc); padding (0) sorts after every candidate
          const uint64_t v = tid < mu ? ((uint64_t)myk << 32) | (uint32_t)~(uint32_t)myj : 0ull;
          const uint64_t r = block_sort_desc(v, P, reinterpret_cast<uint64_t*>(col_lo));
          if (tid < mu) ckey[(int)~(uint32_t)r] = tid < need_u ? kCertainKey : 0u;
          __syncthreads();
        }
        taken = ordered_take(
            m, 0, [&](int j) { return ckey[j] == kCertainKey ? 2 : 0; },
            [&](int p, int j) { if (p < K) out[p] = cand[j]; }, s_eq, s_gt);
      } else {
        int need;
        const uint32_t T = radix_threshold(
            m, K, [&](int j) { return ckey[j]; }, hist, scratch, r_key, s_misc, a.status, &need);
        taken = ordered_take(
            m, need,
            [&](int j) { const uint32_t k = ckey[j]; return k > T ? 2 : (k == T ? 1 : 0); },
            [&](int p, int j) { if (p < K) out[p] = cand[j]; }, s_eq, s_gt);
      }
      if (tid == 0) {
        a.nsel[lr] = K;
        if (taken != K) flag_status(a.status, kStatusCheck);
      }
      finish();
      return;
    }
    // Too many candidates (e.g. heavy ties): canonical scores for the whole row.
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const bool adm = s0[i] != kMinusInfBits;
      s0[i] = adm ? __float_as_uint(canonical_score(qf, kbase + (size_t)ui[i] * 128, wf, a.Hh))
                  : kMinusInfBits;
    }
    __syncthreads();
    canonical = true;
  }

  if (canonical) {
    int need;
    auto key_at = [&](int i) {
      const uint32_t b = s0[i];
      return b == kMinusInfBits ? kNoScoreKey : score_key(__uint_as_float(b));
    };
    const uint32_t T = radix_threshold(n, K, key_at, hist, scratch, r_key, s_misc, a.status, &need);
    const int taken = ordered_take(
        n, need, [&](int i) { const uint32_t k = key_at(i); return k > T ? 2 : (k == T ? 1 : 0); },
        [&](int p, int i) { if (p < K) out[p] = ui[i]; }, s_eq, s_gt);
    if (tid == 0) {
      a.nsel[lr] = K;
      if (taken != K) flag_status(a.status, kStatusCheck);
    }
  }
  finish();
}

template <int NCH, int HH>
cudaError_t launch_tc(const SelDims& d, const ScoreArgs& a, cudaStream_t s) {
  const size_t smem = TcGeom<NCH>::kSmem;
  ScoreArgs ta = a;
  ta.tma = key_tile_map(&ta.kmap, a.keys, d.N, d.L, d.key_stride, 128) == cudaSuccess ? 1 : 0;
  cudaError_t err = cudaFuncSetAttribute(k5_score_tc<NCH, HH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // One persistent CTA per SM; each takes a contiguous range of the union tiles.
  const long long tiles = (long long)((d.N + 127) / 128) * d.L;
  int grid = device_sm_count();
  if (tiles < grid) grid = (int)tiles;
  if (grid < 1) grid = 1;
  // a programmatic dependent of the compaction: the CTAs set up while it finishes
  return launch_pdl(k5_score_tc<NCH, HH>, dim3(grid), TcGeom<NCH>::kThreads, smem, s, ta);
}

}  // namespace

SelLayout sel_layout(const SelDims& d, bool caller_cidx) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t LR = (size_t)d.L * d.R;
  const size_t W = (size_t)(d.N + 31) / 32;
  SelLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  L.uagg = off; off += up(sizeof(uint32_t) * (size_t)d.L * ((W + kCompactThreads - 1) / kCompactThreads));
  L.ldone = off; off += up(sizeof(uint32_t) * (size_t)d.L);
  L.zero_bytes = off;
  L.wordoff = off; off += up(sizeof(int32_t) * (size_t)d.L * W);
  if (!caller_cidx) {
    L.cidx = off; off += up(sizeof(int32_t) * LR * (size_t)d.N);
    L.ccount = off; off += up(sizeof(int32_t) * LR);
  } else {
    L.cidx = L.ccount = (size_t)-1;
  }
  L.uidx = off; off += up(sizeof(int32_t) * (size_t)d.L * d.N);
  L.ucount = off; off += up(sizeof(int32_t) * (size_t)d.L);
  L.urows = off; off += up((size_t)d.L * d.N);
  L.cscore = off; off += up(sizeof(float) * LR * (size_t)score_stride(d.N));
  L.knorm = off; off += up(sizeof(float) * (size_t)d.L * score_stride(d.N));
  L.kmax = off; off += up(sizeof(float) * (size_t)d.L * chunk_stride(d.N));
  L.qnorm = off; off += up(sizeof(float) * LR);
  L.smax = off; off += up(sizeof(float) * LR * (size_t)chunk_stride(d.N));
  L.total = off;
  return L;
}

bool tc_scoring_supported(const SelDims& d, const uint16_t* keys, const uint16_t* q) {
  const int RH = d.R * d.Hh;
  return RH <= 128 && d.D == 128 && (reinterpret_cast<uintptr_t>(keys) % 16) == 0 &&
         (reinterpret_cast<uintptr_t>(q) % 16) == 0 && (d.key_stride % 8) == 0 && d.R <= 8;
}

cudaError_t launch_compact(const SelDims& d, const uint32_t* mask, const int32_t* limit,
                           const SelWorkspace& ws, bool want_cidx, cudaStream_t s) {
  CompactArgs a{d.L, d.R, d.N, mask, limit, ws.cidx, ws.ccount, ws.uidx, ws.ucount, ws.urows,
                ws.wordoff, ws.uagg, ws.header, d.topk, want_cidx ? 1 : 0};
  const int W = (d.N + 31) / 32;
  const int P = (W + kCompactThreads - 1) / kCompactThreads;
  k6_compact<<<d.L * d.R + d.L * P, kCompactThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_score(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                         const float* head_w, const uint32_t* mask, const int32_t* limit,
                         const SelWorkspace& ws, bool tc, cudaStream_t s) {
  ScoreArgs a{d.L, d.R, d.Hh, d.N, d.key_stride, keys, q, head_w, mask, limit, ws.uidx,
              ws.ucount, ws.urows, ws.wordoff, reinterpret_cast<uint32_t*>(ws.cscore), ws.knorm,
              ws.qnorm, ws.kmax, ws.header};
  a.NS = score_stride(d.N);
  a.NC = chunk_stride(d.N);
  a.smax = ws.smax;
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
  const int nch = (d.R * d.Hh + 15) / 16;
  if (d.Hh == 8) {   // the common index-head count gets a static epilogue
    switch (nch) {
      case 1: return launch_tc<1, 8>(d, a, s);
      case 2: return launch_tc<2, 8>(d, a, s);
      case 3: return launch_tc<3, 8>(d, a, s);
      case 4: return launch_tc<4, 8>(d, a, s);
    }
  }
  switch (nch) {
    case 1: return launch_tc<1, 0>(d, a, s);
    case 2: return launch_tc<2, 0>(d, a, s);
    case 3: return launch_tc<3, 0>(d, a, s);
    case 4: return launch_tc<4, 0>(d, a, s);
    case 5: return launch_tc<5, 0>(d, a, s);
    case 6: return launch_tc<6, 0>(d, a, s);
    case 7: return launch_tc<7, 0>(d, a, s);
    case 8: return launch_tc<8, 0>(d, a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                        const float* head_w, int32_t* sel, int32_t* nsel,
                        const SelWorkspace& ws, bool tc, bool keep, cudaStream_t s) {
  TopkArgs a{d.R, d.Hh, d.N, d.topk, d.key_stride, keys, q, head_w, ws.cidx, ws.ccount,
             ws.uidx, ws.ucount, reinterpret_cast<uint32_t*>(ws.cscore), ws.knorm, ws.qnorm,
             ws.kmax, sel, nsel, ws.header, tc ? 1 : 0};
  a.NS = score_stride(d.N);
  a.NC = chunk_stride(d.N);
  a.ldone = ws.ldone;
  a.urows = ws.urows;
  a.keep = keep ? 1 : 0;
  a.smax = ws.smax;
  cudaError_t err =
      cudaFuncSetAttribute(k7_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTopkSmem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k7_topk, d.L * d.R, kTopkThreads, kTopkSmem, s, a);
}

}  // namespace dsmoe
