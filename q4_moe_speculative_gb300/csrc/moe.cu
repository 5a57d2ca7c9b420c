// moe.cu — the speculative-verify Q4 MoE layer: router (K1), gate+up+SwiGLU (K3) and the
// down projection with the rank-ordered combine in its epilogue (K4); the conversion of Q4
// weights to the tile-major layout the kernels stream (K0).
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)".
//   paragraph "Decode": the 384-expert router is one dispatch; the shared expert's
//     gate+up+SwiGLU is one kernel; BF16 rounding happens inside the producing kernels.
//   paragraph "DSpark": the decode step is a 6-row verify and the rows share one weight
//     stream.
//
// Every Q4 weight byte of the shared expert and of the union of routed experts is loaded
// from HBM once per call and applied to every row that uses it. All reductions run in a
// fixed order that does not depend on R or on the other rows, so an R-row call writes the
// same bytes as R one-row calls.
//
// Weights are streamed in the tile-major layout (written once by K0 from the planar Q4
// format): a tile is 16 rows x 64 values (two Q4 blocks) in 576 bytes, the 512 bytes of
// nibbles in the order the tensor-core fragments want them (lane L = 4g + q holds word q of
// rows g and g + 8 of both blocks in its 16 bytes) followed by the 64 bytes of fp16 scales
// (8 bytes per row pair g, g + 8). Tiles run along K within a 16-row tile row, tile rows
// follow one another (in groups of 16 tile rows, K tile first within a group, for the
// down matrices). A pipeline stage is therefore one or two long contiguous runs,
// moved by 1D bulk copies at the full HBM rate, and every fragment read from shared memory
// is one conflict-free 16-byte load.
//
// Q4 dot products run on the tensor cores as mma.sync m16n8k16 (bf16 in, fp32 accumulate)
// with the weights dequantised in registers: the M dimension is 16 weight rows, N = 8 is the
// (up to 6) verify rows, K = 16 values of one 32-value Q4 block, so each block's fp16 scale
// is applied exactly to that block's two MMAs. Widening a 32-bit word of 8 nibbles costs
// three shifts, four AND-ORs that put nibbles in the mantissa of the bf16 number
// 128 + nibble, and four bf16x2 subtractions of 136 (exact q = nibble - 8).
#include <climits>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace dsmoe {
namespace {

using namespace sm100;

// Pipeline waits sleep in polls of at most kWaitSleepNs and give up after kWaitPolls polls
// (about 1 s in all).
#ifndef DSMOE_WAIT_SLEEP_NS
#define DSMOE_WAIT_SLEEP_NS 2000
#endif
constexpr uint32_t kWaitSleepNs = DSMOE_WAIT_SLEEP_NS;
constexpr uint32_t kWaitPolls = kWaitSleepNs > 0 ? (1u << 30) / kWaitSleepNs : (1u << 20);

__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity) {
  if constexpr (kWaitSleepNs > 0)
    return mbar_wait_sleep(bar, parity, kWaitPolls, kWaitSleepNs);
  else
    return mbar_wait(bar, parity, kWaitPolls);
}
constexpr int kTile = kQ4TileBytes;         // 576: 16 rows x 64 values
constexpr int kTileNib = 512;               // nibble bytes of a tile; the scales follow

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- PTX helpers --------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte async copy global -> shared.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// 1D bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-aligned),
// completing `bytes` of the transaction count of `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// bf16 pair (q_lo, q_hi) of the nibbles at bits 0-3 and 16-19 of w: (w & 0x000F000F) |
// 0x43004300 is the bf16 pair (128 + n_lo, 128 + n_hi); minus 136 gives n - 8 exactly.
__device__ __forceinline__ uint32_t q4_pair(uint32_t w) {
  uint32_t p, d;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(p) : "r"(w));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(p), "r"(0x43084308u));
  return d;
}

// D = A (16x16 bf16) * B (16x8 bf16) + C, fp32.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// One Q4 block for the 16 rows of a tile: w_lo / w_hi are word q (values 8q..8q+7 of the
// block) of rows g and g+8 of this lane (g = lane/4, q = lane%4); X holds the matching
// activations of verify row g as bf16 pairs (v0,v4),(v1,v5),(v2,v6),(v3,v7). The block's
// two MMAs use the K order (8q+0, 8q+4 | 8q+1, 8q+5) and (8q+2, 8q+6 | 8q+3, 8q+7), a
// permutation within the block shared by A and B. Returns the raw block dot products
// D[row g / g+8][col 2q, 2q+1] (before the block scale).
__device__ __forceinline__ void q4_block_mma(uint32_t w_lo, uint32_t w_hi, const uint4& X,
                                             float (&d)[4]) {
  const float z[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t p0 = q4_pair(w_lo), p1 = q4_pair(w_lo >> 4);
  const uint32_t r0 = q4_pair(w_hi), r1 = q4_pair(w_hi >> 4);
  mma16816(d, p0, r0, p1, r1, X.x, X.y, z);
  const uint32_t p2 = q4_pair(w_lo >> 8), p3 = q4_pair(w_lo >> 12);
  const uint32_t r2 = q4_pair(w_hi >> 8), r3 = q4_pair(w_hi >> 12);
  mma16816(d, p2, r2, p3, r3, X.z, X.w, d);
}

// acc (rows g, g+8 of this lane) += scale * the raw block dot products d.
__device__ __forceinline__ void scale_add(float (&acc)[4], float s_g, float s_g8,
                                          const float (&d)[4]) {
  acc[0] = __fmaf_rn(s_g, d[0], acc[0]);
  acc[1] = __fmaf_rn(s_g, d[1], acc[1]);
  acc[2] = __fmaf_rn(s_g8, d[2], acc[2]);
  acc[3] = __fmaf_rn(s_g8, d[3], acc[3]);
}

// Both blocks of one tile for this lane: W = the lane's 16 nibble bytes, S = the 8 bytes of
// scales of its row pair, X0 / X1 the activations of the tile's two blocks.
__device__ __forceinline__ void q4_tile_mma(const uint4& W, const uint2& S, const uint4& X0,
                                            const uint4& X1, float (&acc)[4]) {
  const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(&S.x));   // block 0
  const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(&S.y));   // block 1
  float d[4];
  q4_block_mma(W.x, W.y, X0, d);
  scale_add(acc, s0.x, s0.y, d);
  q4_block_mma(W.z, W.w, X1, d);
  scale_add(acc, s1.x, s1.y, d);
}

// Natural-order bf16 values v0..v7 (as 4 packed words) -> MMA pair order.
__device__ __forceinline__ uint4 pair_order(const uint4& v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                    __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint2 lds64(const uint8_t* p) {
  return *reinterpret_cast<const uint2*>(p);
}

// ---------------------------------------------------------------------------------
// K0: planar Q4 -> tile-major. One thread per (tile, lane): the lane's 16 bytes of nibble
// words (word q of rows g and g + 8, blocks 2u and 2u + 1 of the tile's K range), and for
// lanes 0..7 the 8 bytes of scales of row pair (lane, lane + 8). Tile rows are ordered in
// groups of G: within a group (the last one of a matrix may be shorter), by K tile first,
// then by tile row, so that G tile rows x a few K tiles are one contiguous run.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k0_q4_tile(const uint8_t* __restrict__ qs,
                                                  const uint16_t* __restrict__ sc,
                                                  int64_t tiles, int TR, int T, int K, int G,
                                                  uint8_t* __restrict__ dst) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tile = i >> 5;
  if (tile >= tiles) return;
  const int lane = (int)(i & 31), g = lane >> 2, q = lane & 3;
  const int64_t trg = tile / T;                   // tile row over all matrices
  const int u = (int)(tile - trg * T);
  const int64_t mat = trg / TR;
  const int t = (int)(trg - mat * TR);            // tile row within the matrix
  const int g0 = t / G * G, rig = min(G, TR - g0);
  const int64_t out = (mat * TR + g0) * T + (int64_t)u * rig + (t - g0);
  const size_t row_qs = (size_t)K / 2, row_sc = (size_t)K / 32;
  const uint8_t* p0 = qs + (size_t)(trg * 16 + g) * row_qs + (size_t)u * 32 + q * 4;
  const uint8_t* p1 = p0 + 8 * row_qs;
  uint4 v;
  v.x = *reinterpret_cast<const uint32_t*>(p0);        // row g,     block 2u
  v.y = *reinterpret_cast<const uint32_t*>(p1);        // row g + 8, block 2u
  v.z = *reinterpret_cast<const uint32_t*>(p0 + 16);   // row g,     block 2u + 1
  v.w = *reinterpret_cast<const uint32_t*>(p1 + 16);   // row g + 8, block 2u + 1
  uint8_t* tp = dst + (size_t)out * kTile;
  *reinterpret_cast<uint4*>(tp + lane * 16) = v;
  if (lane < 8) {
    const uint16_t* s0 = sc + (size_t)(trg * 16 + lane) * row_sc + 2 * u;
    const uint16_t* s1 = s0 + 8 * row_sc;
    uint2 sv;
    sv.x = (uint32_t)s0[0] | ((uint32_t)s1[0] << 16);
    sv.y = (uint32_t)s0[1] | ((uint32_t)s1[1] << 16);
    *reinterpret_cast<uint2*>(tp + kTileNib + lane * 8) = sv;
  }
}

// ---------------------------------------------------------------------------------
// Prologue: zeroes the words of the workspace that must start at zero (status word,
// router arrival count, combine arrival counts) and lets the router start at once; the
// router waits for this grid only before its arrival count.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k0_clear(uint32_t* __restrict__ p, int nwords) {
  pdl_trigger();
  for (int i = threadIdx.x; i < nwords; i += blockDim.x) p[i] = 0u;
}

// ---------------------------------------------------------------------------------
// K1: router. CTA c computes z = x . Wr[e] for two experts e and all R rows: warps 0-3
// take expert 2c, warps 4-7 expert 2c + 1, warp w the (w % 4)-th quarter of the hidden
// dimension (each lane up to 4 chunks of 8 values, all requested before the first is
// used, x read straight from global memory). A lane adds its chunks in order, the warp's
// lanes are added by a butterfly, the four warps' sums in warp order, and the sigmoid
// score is written. The last CTA to arrive (atomic count, nobody waits) selects each row's
// top k (one warp per row, its scores in registers, a tree argmax per round with ties to
// the lower index), renormalises the weights, and builds the union of the selected
// experts with each one's rows and rank slots.
// ---------------------------------------------------------------------------------
constexpr int kRouterWarps = 8;
constexpr int kRouterExperts = 2;
constexpr int kRouterChunks = 4;   // chunks of 8 values per lane in flight

template <int KPER>   // score registers per lane in the top-k: ceil(E / 32) <= KPER
__global__ void __launch_bounds__(kRouterWarps * 32)
    k1_router(const uint16_t* __restrict__ x, int R, int H, const uint16_t* __restrict__ wr,
              int E, int k, float* __restrict__ scores, int32_t* __restrict__ topk_idx,
              float* __restrict__ topk_w, RouteInfo* __restrict__ route, WsHeader* hdr) {
  __shared__ float part[kRouterWarps][kMaxRows];
  __shared__ int s_is_last;
  __shared__ int32_t sel_e[kMaxRows][kMaxTopK];
  __shared__ float sel_s[kMaxRows][kMaxTopK];
  __shared__ uint32_t ubits[kMaxExperts / 32];
  __shared__ int16_t upos[kMaxExperts];
  __shared__ uint32_t u_rowmask[kMaxUnion];
  __shared__ int8_t u_slot[kMaxUnion][8];
  __shared__ int s_nunion;

  pdl_trigger();   // the gate/up kernel may launch now; it waits for this grid's results
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e = blockIdx.x * kRouterExperts + (warp >> 2);
  {
    float acc[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.0f;
    const int quarter = H / 4;            // a multiple of 16
    const int nch = quarter / 8;
    const int col0 = (warp & 3) * quarter;
    if (e < E) {
      const uint16_t* wrow = wr + (size_t)e * H + col0;
      for (int c0 = lane; c0 < nch; c0 += 32 * kRouterChunks) {
        // every load of the batch (weights, then the rows' activations) is issued before
        // the first multiply, so the batch costs one memory round trip
        uint4 wv[kRouterChunks], xv[kRouterChunks][kMaxRows];
#pragma unroll
        for (int j = 0; j < kRouterChunks; ++j) {
          const int c = min(c0 + 32 * j, nch - 1);
          wv[j] = __ldcs(reinterpret_cast<const uint4*>(wrow + c * 8));
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r)
            xv[j][r] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)min(r, R - 1) * H + col0 + c * 8));
        }
#pragma unroll
        for (int j = 0; j < kRouterChunks; ++j) {
          if (c0 + 32 * j >= nch) break;
          const float wf[8] = {bf16_lo(wv[j].x), bf16_hi(wv[j].x), bf16_lo(wv[j].y),
                               bf16_hi(wv[j].y), bf16_lo(wv[j].z), bf16_hi(wv[j].z),
                               bf16_lo(wv[j].w), bf16_hi(wv[j].w)};
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            const uint4 xr = xv[j][r];
            float t = acc[r];
            t = __fmaf_rn(wf[0], bf16_lo(xr.x), t); t = __fmaf_rn(wf[1], bf16_hi(xr.x), t);
            t = __fmaf_rn(wf[2], bf16_lo(xr.y), t); t = __fmaf_rn(wf[3], bf16_hi(xr.y), t);
            t = __fmaf_rn(wf[4], bf16_lo(xr.z), t); t = __fmaf_rn(wf[5], bf16_hi(xr.z), t);
            t = __fmaf_rn(wf[6], bf16_lo(xr.w), t); t = __fmaf_rn(wf[7], bf16_hi(xr.w), t);
            acc[r] = t;   // rows >= R accumulate a copy of row R - 1, never read
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < R) {
        const float v = warp_sum(acc[r]);
        if (lane == 0) part[warp][r] = v;
      }
    }
  }
  __syncthreads();
  if (tid < kRouterExperts * R) {
    const int ee = tid / R, r = tid - ee * R;
    const int e2 = blockIdx.x * kRouterExperts + ee;
    if (e2 < E) {
      float z = 0.0f;
#pragma unroll
      for (int w = 0; w < 4; ++w) z = __fadd_rn(z, part[ee * 4 + w][r]);
      scores[r * E + e2] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
    }
  }

  // Arrival count: the last CTA continues, the others are done. Nobody waits. (The CTA
  // barrier orders the scores before thread 0's fence, which makes them visible device-wide
  // before the count.) The count was zeroed by the prologue grid, which thread 0 waits for.
  __syncthreads();
  if (tid == 0) {
    pdl_wait();
    __threadfence();
    const unsigned prev = atomicAdd(&hdr->router_arrivals, 1u);
    s_is_last = (prev == gridDim.x - 1);
    if (s_is_last) __threadfence();   // the other CTAs' scores are visible to this CTA after
                                      // the barrier below (the fence is cumulative)
  }
  __syncthreads();
  if (!s_is_last) return;

  if (tid < kMaxExperts / 32) ubits[tid] = 0u;
  if (warp < R) {
    // Row r's top k by (score desc, expert asc): each round takes the warp-wide largest
    // key (one reduction), then the smallest expert index holding it (a second one).
    // Keys: score bits + 2 for a score (sigmoid scores lie in [0, 1], so the bits order
    // like the values), 1 for NaN (from NaN inputs; ranks below every score), 0 for none.
    const int r = warp;
    uint32_t key[KPER];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < KPER; ++i) {
      const int e2 = i * 32 + lane;
      const float sv = e2 < E ? __ldcg(scores + r * E + e2) : 0.0f;
      bad |= (e2 < E) && !(sv >= 0.0f);
      key[i] = e2 >= E ? 0u : (sv >= 0.0f ? __float_as_uint(sv) + 2u : 1u);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(&hdr->status, kStatusCheck);
    for (int j = 0; j < k; ++j) {
      // this lane's largest key and its lowest register index (a tree; ties keep the left)
      uint32_t bk[KPER];
      int bi[KPER];
#pragma unroll
      for (int i = 0; i < KPER; ++i) { bk[i] = key[i]; bi[i] = i; }
#pragma unroll
      for (int w = 1; w < KPER; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < KPER; i += 2 * w)
          if (bk[i + w] > bk[i]) { bk[i] = bk[i + w]; bi[i] = bi[i + w]; }
      const uint32_t mk = __reduce_max_sync(0xffffffffu, bk[0]);
      const uint32_t widx = __reduce_min_sync(
          0xffffffffu, bk[0] == mk ? (uint32_t)(bi[0] * 32 + lane) : 0xFFFFFFFFu);
#pragma unroll
      for (int i = 0; i < KPER; ++i)
        if ((uint32_t)(i * 32 + lane) == widx) key[i] = 0u;   // taken
      if (lane == 0) {
        sel_e[r][j] = (int32_t)widx;
        sel_s[r][j] = mk >= 2u ? __uint_as_float(mk - 2u) : -1.0f;
      }
    }
    __syncwarp();
    // renormalise: the sum in rank order (one lane), then one division per lane
    float sum = 0.0f;
    if (lane == 0) {
      sum = sel_s[r][0];
      for (int j = 1; j < k; ++j) sum = __fadd_rn(sum, sel_s[r][j]);
    }
    sum = __shfl_sync(0xffffffffu, sum, 0);
    if (lane < k) {
      topk_idx[r * k + lane] = sel_e[r][lane];
      topk_w[r * k + lane] = __fdiv_rn(sel_s[r][lane], sum);
    }
  }
  __syncthreads();

  for (int i = tid; i < R * k; i += blockDim.x) {
    const int e2 = sel_e[i / k][i % k];
    atomicOr(&ubits[e2 >> 5], 1u << (e2 & 31));
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t b = ubits[lane];
    const int c = __popc(b);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int pos = incl - c;
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      const int e2 = lane * 32 + bit;
      upos[e2] = (int16_t)pos;
      route->expert[pos] = e2;
      u_rowmask[pos] = 0u;
#pragma unroll
      for (int r = 0; r < 8; ++r) u_slot[pos][r] = -1;
      ++pos;
    }
    if (lane == 31) s_nunion = incl;
  }
  __syncthreads();
  for (int i = tid; i < R * k; i += blockDim.x) {
    const int r = i / k, j = i % k;
    const int p = upos[sel_e[r][j]];
    atomicOr(&u_rowmask[p], 1u << r);
    u_slot[p][r] = (int8_t)(j + 1);
  }
  __syncthreads();
  const int nu = s_nunion;
  for (int i = tid; i < nu; i += blockDim.x) {
    route->rowmask[i] = u_rowmask[i];
#pragma unroll
    for (int r = 0; r < 8; ++r) route->slot[i][r] = u_slot[i][r];
  }
  if (tid == 0) route->n_union = nu;
}

// ---------------------------------------------------------------------------------
// Weight streaming for K3 and K4. A CTA has 16 consumer warps and one producer warp; a
// ring of stages in shared memory is handed over with "full" and "empty" mbarriers, so the
// copies of the next stages are always in flight while the consumers compute. A stage is a
// few long runs of consecutive tiles, each one 1D bulk copy. Work is assigned statically,
// so the split depends only on the sizes.
// ---------------------------------------------------------------------------------
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kMmaThreads = kConsumers + 32;            // + producer warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMaxRing = 8;
constexpr int kReducerWarps = 3;                         // gate/up: 16 rows x R <= 96 outputs
constexpr int kGuThreads = kMmaThreads + 32 * kReducerWarps;
constexpr int kConsumerBarrier = 1;                     // named barrier id of the consumers
constexpr int kXPad = 64;                                // staged activation row pad (bytes)

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_addr(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(kConsumers) : "memory");
}

// ---------------------------------------------------------------------------------
// K3: gate + up + SwiGLU. A unit is (expert slot u, tile row of I = 16 rows): slot 0 is the
// shared expert (all rows), slot u >= 1 the u-th expert of the union (its rows). CTA b
// takes units b, b + G, b + 2G, ... (G = grid). A stage is one K chunk of a unit: CT
// consecutive tiles of the gate tile row and the same of the up tile row, two bulk copies.
// Consumer warp w takes tiles CT/16 w .. CT/16 w + CT/16 - 1 of the chunk for both matrices
// and keeps its partial sums across the unit's chunks. At the end of a unit the 16 warps'
// partials meet in shared memory and are added in warp order by the reducer warps, which
// write h = bf16_rne(silu(g) * u) for the expert's rows. The activations sit in shared
// memory as bf16 in MMA pair order, staged once per CTA while the router runs; the
// producer starts on the shared expert's units before the router's results exist.
// ---------------------------------------------------------------------------------
struct GateUpArgs {
  const uint8_t* gate;     // tiles [E][I/16][H/64]
  const uint8_t* up;
  const uint8_t* sh_gate;  // tiles [I/16][H/64]
  const uint8_t* sh_up;
  const uint16_t* x;
  const RouteInfo* route;
  uint16_t* h;
  uint32_t* status;
  int R, H, I, k, ring;
};

__host__ __device__ constexpr size_t gu_red_bytes(int R) {
  return 2ull * kConsumerWarps * 2 * 16 * (size_t)R * 4;
}
template <int CT>
__host__ __device__ constexpr size_t gu_stage_bytes() { return 2ull * CT * kTile; }

template <int CT>   // tiles per matrix per stage: 32 or 16
__global__ void __launch_bounds__(kGuThreads, 1) k3_gate_up(const GateUpArgs a) {
  constexpr int TPW = CT / kConsumerWarps;   // tiles per warp per matrix per stage
  constexpr int kStage = (int)gu_stage_bytes<CT>();
  __shared__ __align__(8) uint64_t full[kMaxRing], empty[kMaxRing];
  // partial-sum buffers: written by the 16 consumer warps (pfull), read by the reducer
  // warps (pempty); two buffers, so consumers wait only when two units are unreduced
  __shared__ __align__(8) uint64_t s_pfull[2], s_pempty[2];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int R = a.R, H = a.H, I = a.I, k = a.k, ring = a.ring;
  const int T = H >> 6;                           // tiles per tile row (K = H)
  const int KC = (T + CT - 1) / CT;               // chunks per unit
  const int RT = I >> 4;                          // tile rows (units) per expert
  const size_t expert_bytes = (size_t)RT * T * kTile;
  const int xstride = 2 * H + kXPad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;

  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)ring * kStage);
  uint8_t* xs = smem + (size_t)ring * kStage + gu_red_bytes(R);

  if (tid == 0) {
    for (int s = 0; s < ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_pfull[b], kConsumerWarps);
      mbar_init(&s_pempty[b], kReducerWarps);
    }
    fence_mbar_init();
  }
  // Activations -> shared memory, bf16 in MMA pair order (independent of the router).
#pragma unroll 4
  for (int i = tid; i < R * (H >> 3); i += blockDim.x) {
    const int r = i / (H >> 3), grp = i - r * (H >> 3);
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + (size_t)r * H + grp * 8);
    *reinterpret_cast<uint4*>(xs + r * xstride + (grp >> 2) * 64 + (grp & 3) * 16) = pair_order(v);
  }
  __syncthreads();

  const int G = gridDim.x;
  bool timed_out = false;
  if (warp == kProducerWarp) {
    bool routed = false;   // the router's results are known to be visible
    // Units of the shared expert need nothing from the router; a unit of a routed expert
    // waits for it (and so does the count of units, which needs the union size).
    int slot = 0, f = 0;
    uint32_t phase = 0;    // ring cursor: stage f sits in `slot`, pass parity `phase`
    for (int n = (int)blockIdx.x;; n += G) {
      const int u = n / RT, rt = n - u * RT;
      if (u > 0 && !routed) { pdl_wait(); routed = true; }
      if (routed && n >= (1 + a.route->n_union) * RT) break;
      const uint8_t* gbase = (u == 0 ? a.sh_gate : a.gate + (size_t)a.route->expert[u - 1] * expert_bytes) +
                             (size_t)rt * T * kTile;
      const uint8_t* ubase = (u == 0 ? a.sh_up : a.up + (size_t)a.route->expert[u - 1] * expert_bytes) +
                             (size_t)rt * T * kTile;
      for (int c = 0; c < KC; ++c, ++f) {
        if (f >= ring && !pipe_wait(&empty[slot], phase ^ 1u)) timed_out = true;
        if (lane == 0) {
          uint8_t* st = stages + (size_t)slot * kStage;
          const uint32_t bytes = (uint32_t)min(CT, T - c * CT) * kTile;
          mbar_arrive_expect_tx(&full[slot], 2u * bytes);
          bulk_copy(st, gbase + (size_t)c * CT * kTile, bytes, &full[slot]);
          bulk_copy(st + CT * kTile, ubase + (size_t)c * CT * kTile, bytes, &full[slot]);
        }
        __syncwarp();
        if (++slot == ring) { slot = 0; phase ^= 1u; }
      }
    }
    if (!routed) pdl_wait();
  } else if (warp < kProducerWarp) {
    pdl_wait();      // the route produced by the router grid is visible from here on
    const RouteInfo* rt = a.route;
    const int n_units = (1 + rt->n_union) * RT;
    const int n_mine = (int)blockIdx.x < n_units ? (n_units - (int)blockIdx.x + G - 1) / G : 0;
    const uint8_t* xrow = xs + min(g, R - 1) * xstride + q * 16;   // rows >= R: any finite row
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    int slot = 0;
    uint32_t phase = 0;
    for (int unit = 0; unit < n_mine; ++unit) {
      for (int c = 0; c < KC; ++c) {
        if (!pipe_wait(&full[slot], phase)) timed_out = true;
        const uint8_t* st = stages + (size_t)slot * kStage;
        const int ct = min(CT, T - c * CT);
        const uint8_t* xc = xrow + (size_t)c * CT * 128;
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt) {
          const int t = warp * TPW + tt;
          if (t < ct) {
            const uint8_t* xb = xc + t * 128;   // blocks 2t, 2t + 1 of the chunk
            const uint4 X0 = lds128(xb), X1 = lds128(xb + 64);
            const uint8_t* tg = st + t * kTile;
            const uint8_t* tu = st + (CT + t) * kTile;
            const uint4 Wg = lds128(tg + lane * 16), Wu = lds128(tu + lane * 16);
            const uint2 Sg = lds64(tg + kTileNib + g * 8), Su = lds64(tu + kTileNib + g * 8);
            q4_tile_mma(Wg, Sg, X0, X1, ag);
            q4_tile_mma(Wu, Su, X0, X1, au);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);   // this warp is done with the slot
        if (++slot == ring) { slot = 0; phase ^= 1u; }
      }
      // partials [warp][gate/up][row][col] (cols < R only) into buffer unit & 1, once the
      // reducers are done with the unit that used it before
      const int buf = unit & 1;
      if (unit >= 2 && !pipe_wait(&s_pempty[buf], ((unit >> 1) - 1) & 1)) timed_out = true;
      float* rb = red + (size_t)buf * kConsumerWarps * 2 * 16 * R;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = 2 * q + (e & 1), row = g + ((e & 2) ? 8 : 0);
        if (col < R) {
          rb[((warp * 2 + 0) * 16 + row) * R + col] = ag[e];
          rb[((warp * 2 + 1) * 16 + row) * R + col] = au[e];
        }
        ag[e] = 0.f;
        au[e] = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_pfull[buf]);
    }
  } else {
    // Reducers: for each unit of this CTA, in order, the 16 warps' partials are added in
    // warp order and h = bf16_rne(silu(g) * u) is written for the expert's rows.
    pdl_wait();
    const RouteInfo* rt = a.route;
    const int n_units = (1 + rt->n_union) * RT;
    const int rtid = tid - (kProducerWarp + 1) * 32;
    int unit = 0;
    for (int n = (int)blockIdx.x; n < n_units; n += G, ++unit) {
      const int b = unit & 1;
      if (!pipe_wait(&s_pfull[b], (unit >> 1) & 1)) {
        timed_out = true;
        break;
      }
      const float* rb = red + (size_t)b * kConsumerWarps * 2 * 16 * R;
      const int u = n / RT, rti = n - u * RT;
      if (rtid < 16 * R) {
        const int row = rtid / R, col = rtid - row * R;
        const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : rt->rowmask[u - 1];
        if ((rowmask >> col) & 1u) {
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) {
            gs = __fadd_rn(gs, rb[((w * 2 + 0) * 16 + row) * R + col]);
            us = __fadd_rn(us, rb[((w * 2 + 1) * 16 + row) * R + col]);
          }
          const int slot_c = (u == 0) ? 0 : rt->slot[u - 1][col];
          const float silu = __fdiv_rn(gs, __fadd_rn(1.0f, expf(-gs)));
          a.h[((size_t)col * (1 + k) + slot_c) * I + rti * 16 + row] =
              f32_to_bf16_rne(__fmul_rn(silu, us));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_pempty[b]);
    }
  }
  pdl_trigger();   // the down projection may be scheduled as CTAs of this grid retire
  if (timed_out && lane == 0) flag_status(a.status, kStatusTimeout);
}

// ---------------------------------------------------------------------------------
// K4: down projection and combine. A unit is (expert slot u, row group of 16 tile rows =
// 256 rows of H); consumer warp w owns tile row w of the group for the whole unit, so its
// fp32 sums need no reduction with other warps. A stage is one K chunk of KT tiles of the
// group's 16 tile rows, one contiguous run (the down matrices keep their tile rows in
// groups of 16, K tile first within a group): one bulk copy. CTA b takes a contiguous
// range of units, so consecutive stages mostly belong to one expert and its h (the B
// operand, kept in shared memory in MMA pair order) is reloaded only when the expert
// changes. At the end of a unit each warp writes o[row][slot] (fp32) for the rows that use
// the expert; a counting warp then counts the unit against its row group (fence, atomic
// add) while the consumers go on, and after its last unit the CTA that completed a row
// group (every slot's unit done; nobody waits) writes y = bf16_rne(o_shared +
// sum_j w_j o_j) for the group's rows, j in rank order.
// The weights do not depend on the gate/up kernel, so the producer starts streaming them
// before that kernel has finished; only h waits for it.
// ---------------------------------------------------------------------------------
#ifndef DSMOE_DOWN_KT
#define DSMOE_DOWN_KT 4
#endif
constexpr int kDownKT = DSMOE_DOWN_KT;   // tiles per tile row per stage
constexpr int kGroupRows = kDownGroup;   // tile rows per unit (one per consumer warp)
constexpr int kDownStage = kGroupRows * kDownKT * kTile;   // 36,864 bytes

struct DownArgs {
  const uint8_t* down;      // tiles [E][H/16][I/64]
  const uint8_t* sh_down;   // tiles [H/16][I/64]
  const uint16_t* h;
  const RouteInfo* route;
  const float* topk_w;
  float* opart;             // [R][1+k][H] expert outputs
  uint32_t* counts;         // [ceil(H/256)] units completed per row group (zeroed per call)
  uint16_t* y;
  uint32_t* status;
  int R, H, I, k, ring;
};

__host__ __device__ constexpr int down_hpitch(int I) { return 2 * I + kXPad; }

constexpr int kCountWarp = kProducerWarp + 1;
constexpr int kDownThreads = kMmaThreads + 32;   // + the counting warp
constexpr int kMaxGroupsPerCta = 64;             // row groups a CTA can complete (H <= 16384)

__global__ void __launch_bounds__(kDownThreads, 1) k4_down(const DownArgs a) {
  __shared__ __align__(8) uint64_t full[kMaxRing], empty[kMaxRing];
  // a unit's outputs written (16 consumer warps) / taken over by the counting warp (1)
  __shared__ __align__(8) uint64_t s_udone[2], s_ufree[2];
  __shared__ uint32_t s_rowmask[kMaxUnion];
  __shared__ __align__(8) int8_t s_slot[kMaxUnion][8];
  __shared__ int s_done[kMaxGroupsPerCta];   // row groups this CTA completed
  __shared__ int s_ndone;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int R = a.R, H = a.H, I = a.I, k = a.k, ring = a.ring;
  const int T = I >> 6;                              // tiles per tile row (K = I)
  const int KC = (T + kDownKT - 1) / kDownKT;        // chunks per unit
  const int RTt = H >> 4;                            // tile rows per expert
  const int NGR = (RTt + kGroupRows - 1) / kGroupRows;
  const size_t expert_bytes = (size_t)RTt * T * kTile;
  const int hpitch = down_hpitch(I);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;

  uint8_t* stages = smem;
  uint8_t* hs = smem + (size_t)ring * kDownStage;   // [8][hpitch]

  if (tid == 0) {
    for (int s = 0; s < ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_udone[b], kConsumerWarps);
      mbar_init(&s_ufree[b], 1);
    }
    s_ndone = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // The route was complete before the gate/up kernel passed its own wait, which precedes
  // the launch of this grid; h is waited for below.
  const RouteInfo* rt = a.route;
  const int n_union = rt->n_union;
  const int n_units = (1 + n_union) * NGR;
  const int G = gridDim.x;
  const int u_begin = (int)(((long long)blockIdx.x * n_units) / G);
  const int u_end = (int)(((long long)(blockIdx.x + 1) * n_units) / G);
  bool timed_out = false;

  if (warp == kProducerWarp) {
    int slot = 0, f = 0;
    uint32_t phase = 0;    // ring cursor
    for (int n = u_begin; n < u_end; ++n) {
      const int u = n / NGR, rg = n - u * NGR;
      const int rig = min(kGroupRows, RTt - rg * kGroupRows);   // tile rows in the group
      const uint8_t* gbase = (u == 0 ? a.sh_down : a.down + (size_t)rt->expert[u - 1] * expert_bytes) +
                             (size_t)rg * kGroupRows * T * kTile;
      for (int c = 0; c < KC; ++c, ++f) {
        if (f >= ring && !pipe_wait(&empty[slot], phase ^ 1u)) timed_out = true;
        if (lane == 0) {
          // the group's tiles of K tiles c KT .. c KT + kt - 1: one contiguous run
          const uint32_t bytes = (uint32_t)(min(kDownKT, T - c * kDownKT) * rig * kTile);
          mbar_arrive_expect_tx(&full[slot], bytes);
          bulk_copy(stages + (size_t)slot * kDownStage,
                    gbase + (size_t)c * kDownKT * rig * kTile, bytes, &full[slot]);
        }
        __syncwarp();
        if (++slot == ring) { slot = 0; phase ^= 1u; }
      }
    }
    pdl_wait();
  } else if (warp == kCountWarp) {
    // Counts each finished unit against its row group: once the consumers' outputs of the
    // unit are written (mbarrier, CTA scope), a fence makes them visible device-wide, then
    // the atomic count; the unit that completes a group (1 + n_union units, nobody waits)
    // records it for the combine below.
    pdl_wait();
    int j = 0;
    for (int n = u_begin; n < u_end; ++n, ++j) {
      const int b = j & 1;
      if (!pipe_wait(&s_udone[b], (j >> 1) & 1)) timed_out = true;
      if (lane == 0) {
        const int rg = n % NGR;
        __threadfence();
        const unsigned prev = atomicAdd(&a.counts[rg], 1u);
        if (prev == (unsigned)n_union) {
          __threadfence();
          if (s_ndone < kMaxGroupsPerCta) s_done[s_ndone++] = rg;
          else flag_status(a.status, kStatusCheck);
        }
        mbar_arrive(&s_ufree[b]);
      }
      __syncwarp();
    }
  } else {
    // the union's row masks and rank slots, read every unit, kept in shared memory (the
    // route is visible already, see above)
    for (int i = tid; i < n_union; i += kConsumers) {
      s_rowmask[i] = rt->rowmask[i];
      *reinterpret_cast<uint2*>(s_slot[i]) = *reinterpret_cast<const uint2*>(rt->slot[i]);
    }
    pdl_wait();      // h is complete from here on
    consumer_sync();
    const uint8_t* hrow = hs + g * hpitch + q * 16;   // rows >= R or unused: never read out
    int h_u = -1;       // expert slot whose h is staged
    // two chains: even (acc) and odd (acc2) tiles of the row, added once at the unit end
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    int slot = 0, j = 0;
    uint32_t phase = 0;
    for (int n = u_begin; n < u_end; ++n, ++j) {
      const int u = n / NGR, rg = n - u * NGR;
      const int rig = min(kGroupRows, RTt - rg * kGroupRows);
      const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : s_rowmask[u - 1];
      if (u != h_u) {
        // h of the expert's rows: [verify row][values], 16-byte pieces, then each piece
        // put in MMA pair order in place. Rows that do not use the expert keep stale
        // values; their MMA columns are never read.
        consumer_sync();   // every consumer is done with the previous h
        const int per_row = I / 8;
        for (int p = tid; p < R * per_row; p += kConsumers) {
          const int rr = p / per_row, pp = p - rr * per_row;
          if ((rowmask >> rr) & 1u) {
            const int slot_r = (u == 0) ? 0 : s_slot[u - 1][rr];
            cp_async16(hs + rr * hpitch + pp * 16, a.h + ((size_t)rr * (1 + k) + slot_r) * I + pp * 8);
          }
        }
        cp_async_commit();
        cp_async_wait<0>();
        for (int p = tid; p < R * per_row; p += kConsumers) {
          const int rr = p / per_row, pp = p - rr * per_row;
          if ((rowmask >> rr) & 1u) {
            uint4* hp = reinterpret_cast<uint4*>(hs + rr * hpitch + pp * 16);
            *hp = pair_order(*hp);
          }
        }
        consumer_sync();
        h_u = u;
      }
      const int tr = rg * kGroupRows + warp;              // this warp's tile row
      for (int c = 0; c < KC; ++c) {
        if (!pipe_wait(&full[slot], phase)) timed_out = true;
        const uint8_t* st = stages + (size_t)slot * kDownStage;
        const int kt = min(kDownKT, T - c * kDownKT);
        if (warp < rig) {
          const uint8_t* xc = hrow + (size_t)c * kDownKT * 128;
          static_assert(kDownKT % 2 == 0, "tiles alternate between the two chains");
#pragma unroll
          for (int jj = 0; jj < kDownKT; ++jj) {
            if (jj < kt) {
              const uint8_t* tp = st + (jj * rig + warp) * kTile;
              const uint4 W = lds128(tp + lane * 16);
              const uint2 S = lds64(tp + kTileNib + g * 8);
              const uint8_t* xb = xc + jj * 128;   // blocks 2t, 2t + 1
              if (jj & 1)
                q4_tile_mma(W, S, lds128(xb), lds128(xb + 64), acc2);
              else
                q4_tile_mma(W, S, lds128(xb), lds128(xb + 64), acc);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == ring) { slot = 0; phase ^= 1u; }
      }
      // the unit is done: this warp's rows, once the counting warp has taken over the unit
      // two before (its outputs are counted before new ones are announced)
      const int b = j & 1;
      if (j >= 2 && !pipe_wait(&s_ufree[b], ((j >> 1) - 1) & 1)) timed_out = true;
      if (warp < rig) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = 2 * q + (e & 1), row = tr * 16 + g + ((e & 2) ? 8 : 0);
          if (col < R && ((rowmask >> col) & 1u)) {
            const int slot_c = (u == 0) ? 0 : s_slot[u - 1][col];
            a.opart[((size_t)col * (1 + k) + slot_c) * H + row] = __fadd_rn(acc[e], acc2[e]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = acc2[e] = 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_udone[b]);
    }
  }
  // The row groups whose last unit this CTA counted: every slot's rows are written, so
  // combine them, rank order (all warps of the CTA).
  __syncthreads();
  const int per_group = R * kGroupRows * 16;   // outputs of a full group
  for (int i = tid; i < s_ndone * per_group; i += kDownThreads) {
    const int d = i / per_group, rem = i - d * per_group;
    const int rg = s_done[d];
    const int r0 = rg * kGroupRows * 16;
    const int r = rem / (kGroupRows * 16), row = r0 + (rem - r * (kGroupRows * 16));
    if (row >= H) continue;   // a short last group
    const float* o = a.opart + (size_t)r * (1 + k) * H + row;
    // every load first (one round trip), then the fma chain in rank order
    float ov[kMaxTopK + 1], wv[kMaxTopK];
#pragma unroll
    for (int jj = 0; jj <= kMaxTopK; ++jj) ov[jj] = jj <= k ? __ldcg(o + (size_t)jj * H) : 0.0f;
#pragma unroll
    for (int jj = 0; jj < kMaxTopK; ++jj) wv[jj] = jj < k ? __ldcg(a.topk_w + r * k + jj) : 0.0f;
    float yv = ov[0];
#pragma unroll
    for (int jj = 0; jj < kMaxTopK; ++jj)
      if (jj < k) yv = __fmaf_rn(wv[jj], ov[1 + jj], yv);
    a.y[(size_t)r * H + row] = f32_to_bf16_rne(yv);
  }
  pdl_trigger();
  if (timed_out && lane == 0) flag_status(a.status, kStatusTimeout);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int CT>
size_t gate_up_smem(const MoeDims& d, int ring) {
  return 1024 + (size_t)ring * gu_stage_bytes<CT>() + gu_red_bytes(d.R) +
         (size_t)d.R * (2 * d.H + kXPad);
}

size_t down_smem(const MoeDims& d, int ring) {
  return 1024 + (size_t)ring * kDownStage + (size_t)8 * down_hpitch(d.I);
}

// Deepest ring (kMaxRing .. lo stages) whose shared memory fits; 0 if none does.
#ifndef DSMOE_RING_MAX
#define DSMOE_RING_MAX kMaxRing
#endif
template <typename F>
int pick_ring(F smem_of, int lo = 2, int hi = DSMOE_RING_MAX) {
  for (int ring = hi; ring >= lo; --ring)
    if (smem_of(ring) <= (size_t)device_max_smem_optin()) return ring;
  return 0;
}

template <int CT>
cudaError_t launch_gate_up_ct(const MoeDims& d, GateUpArgs& a, int ring, cudaStream_t s) {
  const size_t smem = gate_up_smem<CT>(d, ring);
  cudaError_t err = set_smem(k3_gate_up<CT>, smem);
  if (err != cudaSuccess) return err;
  a.ring = ring;
  return launch_pdl(k3_gate_up<CT>, device_sm_count(), kGuThreads, smem, s, a);
}

}  // namespace

size_t gate_up_smem_bytes(const MoeDims& d) { return gate_up_smem<16>(d, 2); }

MoeLayout moe_layout(const MoeDims& d) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  MoeLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  const int ngr = ((d.H >> 4) + kGroupRows - 1) / kGroupRows;
  L.counts = off; off += up(sizeof(uint32_t) * (size_t)ngr);
  L.zero_bytes = off;
  L.scores = off; off += up(sizeof(float) * (size_t)d.R * d.E);
  L.route = off; off += up(sizeof(RouteInfo));
  L.h = off; off += up(sizeof(uint16_t) * (size_t)d.R * (1 + d.k) * d.I);
  L.opart = off; off += up(sizeof(float) * (size_t)d.R * (1 + d.k) * d.H);
  L.total = off;
  return L;
}

cudaError_t launch_tile(const uint8_t* qs, const uint16_t* sc, int n_mats, int64_t rows,
                        int K, int group, uint8_t* dst, cudaStream_t s) {
  const int T = K / 64;
  const int64_t TR = rows / 16;
  const int64_t tiles = (int64_t)n_mats * TR * T;
  const int64_t threads = tiles * 32;
  const int64_t grid = (threads + 255) / 256;
  if (grid <= 0) return cudaSuccess;
  if (grid > INT_MAX || TR > INT_MAX) return cudaErrorInvalidValue;
  k0_q4_tile<<<(unsigned)grid, 256, 0, s>>>(qs, sc, tiles, (int)TR, T, K, group, dst);
  return cudaGetLastError();
}

cudaError_t launch_router(const MoeDims& d, const uint16_t* x, const uint16_t* router_w,
                          int32_t* topk_idx, float* topk_w, const MoeWorkspace& ws,
                          cudaStream_t s) {
  // zero the header and the combine counts (a plain launch: it follows the stream's earlier
  // work), then the router, which overlaps it
  k0_clear<<<1, 256, 0, s>>>(ws.header, (int)(ws.zero_bytes / 4));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int grid = (d.E + kRouterExperts - 1) / kRouterExperts;
  auto* hdr = reinterpret_cast<WsHeader*>(ws.header);
  if (d.E <= 12 * 32)
    return launch_pdl(k1_router<12>, grid, kRouterWarps * 32, 0, s, x, d.R, d.H, router_w, d.E,
                      d.k, ws.scores, topk_idx, topk_w, ws.route, hdr);
  return launch_pdl(k1_router<kMaxExperts / 32>, grid, kRouterWarps * 32, 0, s, x, d.R, d.H,
                    router_w, d.E, d.k, ws.scores, topk_idx, topk_w, ws.route, hdr);
}

cudaError_t launch_gate_up(const MoeDims& d, const uint16_t* x, const uint8_t* gate,
                           const uint8_t* up, const uint8_t* sh_gate, const uint8_t* sh_up,
                           const MoeWorkspace& ws, cudaStream_t s) {
  GateUpArgs a{};
  a.gate = gate; a.up = up; a.sh_gate = sh_gate; a.sh_up = sh_up;
  a.x = x; a.route = ws.route; a.h = ws.h; a.status = ws.header;
  a.R = d.R; a.H = d.H; a.I = d.I; a.k = d.k;
  // Chunks of 32 tiles when a ring of at least 3 of them fits, else chunks of 16.
#ifndef DSMOE_GU_CT
#define DSMOE_GU_CT 32
#endif
  const int ring32 = DSMOE_GU_CT == 32 ? pick_ring([&](int r) { return gate_up_smem<32>(d, r); }, 3) : 0;
  if (ring32) return launch_gate_up_ct<32>(d, a, ring32, s);
  const int ring16 = pick_ring([&](int r) { return gate_up_smem<16>(d, r); });
  if (ring16) return launch_gate_up_ct<16>(d, a, ring16, s);
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_down(const MoeDims& d, const uint8_t* down, const uint8_t* sh_down,
                        const float* topk_w, uint16_t* y, const MoeWorkspace& ws,
                        cudaStream_t s) {
  const int ring = pick_ring([&](int r) { return down_smem(d, r); });
  if (ring == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = down_smem(d, ring);
  cudaError_t err = set_smem(k4_down, smem);
  if (err != cudaSuccess) return err;
  DownArgs a{};
  a.down = down; a.sh_down = sh_down; a.h = ws.h; a.route = ws.route; a.topk_w = topk_w;
  a.opart = ws.opart; a.counts = ws.counts; a.y = y; a.status = ws.header;
  a.R = d.R; a.H = d.H; a.I = d.I; a.k = d.k; a.ring = ring;
  return launch_pdl(k4_down, device_sm_count(), kDownThreads, smem, s, a);
}

}  // namespace dsmoe
