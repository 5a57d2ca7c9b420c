// moe.cu — the speculative-verify Q4 MoE layer: router (K1), gate+up+SwiGLU (K3), down
// projection (K4) and the rank-ordered combine (K5).
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
// Q4 dot products (K3, K4) run on the tensor cores as mma.sync m16n8k16 (bf16 in, fp32
// accumulate) with the weights dequantised in registers: the M dimension is 16 weight rows,
// N = 8 is the (up to 6) verify rows, K = 16 values of one 32-value Q4 block, so each
// block's fp16 scale is applied exactly to that block's two MMAs. Widening a 32-bit word
// of 8 nibbles costs three shifts, four AND-ORs that put nibbles in the mantissa of the
// bf16 number 128 + nibble, and four bf16x2 subtractions of 136 (exact q = nibble - 8).
// A producer warp streams the weights into a ring of CTA-wide stages completed by
// mbarriers: as TMA boxes (a 3D view of the nibbles, [128-byte chunk][row][128 bytes],
// with the 128-byte swizzle, and a 2D box of the scales) when the rows are whole 128-byte
// chunks and the scales 16-byte aligned, else as per-row 1D bulk copies of up to 1 KB and
// 4-byte scale copies.
#include <climits>
#include <utility>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace dsmoe {
namespace {

using namespace sm100;

constexpr int kRouterWarps = 8;
constexpr uint32_t kWaitPolls = 1u << 20;   // bounded mbarrier waits (~1 s)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- PTX helpers --------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte async copy global -> shared; zero-fill (no global read) when !valid.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// The mbarrier receives one arrival once all of this thread's earlier cp.async copies have
// landed; the arrival is counted in the barrier's initial count (noinc).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
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

// Natural-order bf16 values v0..v7 (as 4 packed words) -> MMA pair order.
__device__ __forceinline__ uint4 pair_order(const uint4& v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                    __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

// Four packed fp16 scales (blocks j = 0..3) -> fp32.
__device__ __forceinline__ void widen_scales(uint2 s, float (&f)[4]) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&s.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&s.y));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// ---------------------------------------------------------------------------------
// K1: router. CTA c computes z = x . Wr[e] for the kRouterExperts experts e of its group
// and all R rows: warp w takes the w-th eighth of the hidden dimension (x read straight
// from global memory into registers, each lane 8 values at a time), the eight warps'
// partial sums (lane-strided then a butterfly) are added in warp order, and the sigmoid
// score is written. The last CTA to arrive (atomic count, nobody waits) selects each
// row's top k (one warp per row, its scores in registers, a tree argmax per round with
// ties to the lower index), renormalises the weights, and builds the union of the
// selected experts with each one's rows and rank slots.
// ---------------------------------------------------------------------------------
constexpr int kRouterExperts = 4;

template <int KPER>   // score registers per lane in the top-k: ceil(E / 32) <= KPER
__global__ void __launch_bounds__(kRouterWarps * 32)
    k1_router(const uint16_t* __restrict__ x, int R, int H, const uint16_t* __restrict__ wr,
              int E, int k, float* __restrict__ scores, int32_t* __restrict__ topk_idx,
              float* __restrict__ topk_w, RouteInfo* __restrict__ route, WsHeader* hdr) {
  __shared__ float part[kRouterWarps][kRouterExperts][kMaxRows];
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
  const int e0 = blockIdx.x * kRouterExperts;
  const int ne = min(kRouterExperts, E - e0);
  {
    float acc[kRouterExperts][kMaxRows];
#pragma unroll
    for (int e = 0; e < kRouterExperts; ++e)
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) acc[e][r] = 0.0f;
    const int slice = H / kRouterWarps;          // a multiple of 8
    const int nch = slice / 8;
    // the weights of two chunks per lane are requested before either is used
    for (int c0 = lane; c0 < nch; c0 += 64) {
      uint4 wv2[2][kRouterExperts];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = c0 + 32 * cc, col = warp * slice + c * 8;
#pragma unroll
        for (int e = 0; e < kRouterExperts; ++e)
          wv2[cc][e] = (c < nch && e < ne)
                           ? __ldcs(reinterpret_cast<const uint4*>(wr + (size_t)(e0 + e) * H + col))
                           : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = c0 + 32 * cc;
        if (c >= nch) break;
        const int col = warp * slice + c * 8;
        const uint4* wv = wv2[cc];
        uint4 xv[kMaxRows];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
          xv[r] = r < R ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)r * H + col))
                        : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          if (r < R) {
            const float xf[8] = {bf16_lo(xv[r].x), bf16_hi(xv[r].x), bf16_lo(xv[r].y),
                                 bf16_hi(xv[r].y), bf16_lo(xv[r].z), bf16_hi(xv[r].z),
                                 bf16_lo(xv[r].w), bf16_hi(xv[r].w)};
#pragma unroll
            for (int e = 0; e < kRouterExperts; ++e) {
              float t = acc[e][r];
              t = __fmaf_rn(bf16_lo(wv[e].x), xf[0], t); t = __fmaf_rn(bf16_hi(wv[e].x), xf[1], t);
              t = __fmaf_rn(bf16_lo(wv[e].y), xf[2], t); t = __fmaf_rn(bf16_hi(wv[e].y), xf[3], t);
              t = __fmaf_rn(bf16_lo(wv[e].z), xf[4], t); t = __fmaf_rn(bf16_hi(wv[e].z), xf[5], t);
              t = __fmaf_rn(bf16_lo(wv[e].w), xf[6], t); t = __fmaf_rn(bf16_hi(wv[e].w), xf[7], t);
              acc[e][r] = t;
            }
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < kRouterExperts; ++e)
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < R) {
          const float v = warp_sum(acc[e][r]);
          if (lane == 0) part[warp][e][r] = v;
        }
      }
  }
  __syncthreads();
  if (tid < ne * R) {
    const int e = tid / R, r = tid - e * R;
    float z = 0.0f;
#pragma unroll
    for (int w = 0; w < kRouterWarps; ++w) z = __fadd_rn(z, part[w][e][r]);
    scores[r * E + e0 + e] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
  }

  // Arrival count: the last CTA continues, the others are done. Nobody waits. (The CTA
  // barrier orders the scores before thread 0's fence, which makes them visible device-wide
  // before the count.)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&hdr->router_arrivals, 1u);
    s_is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();

  if (tid < kMaxExperts / 32) ubits[tid] = 0u;
  if (warp < R) {
    const int r = warp;
    float v[KPER];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < KPER; ++i) {
      const int e2 = i * 32 + lane;
      const float sv = e2 < E ? __ldcg(scores + r * E + e2) : -1.0f;
      // sigmoid scores lie in [0, 1]; a NaN (from NaN inputs) ranks below every score
      bad |= (e2 < E) && !(sv >= 0.0f);
      v[i] = (e2 >= E || sv >= 0.0f) ? sv : -0.5f;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(&hdr->status, kStatusCheck);
    for (int j = 0; j < k; ++j) {
      // this lane's best (value, register index) by a tree; on equal values the lower
      // index (the left operand) wins
      float bv[KPER];
      int bi[KPER];
#pragma unroll
      for (int i = 0; i < KPER; ++i) { bv[i] = v[i]; bi[i] = i; }
#pragma unroll
      for (int w = 1; w < KPER; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < KPER; i += 2 * w)
          if (bv[i + w] > bv[i]) { bv[i] = bv[i + w]; bi[i] = bi[i + w]; }
      float best = bv[0];
      int bidx = bi[0] * 32 + lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ov > best || (ov == best && oi < bidx)) { best = ov; bidx = oi; }
      }
#pragma unroll
      for (int i = 0; i < KPER; ++i)
        if (i * 32 + lane == bidx) v[i] = -1.0f;   // taken
      if (lane == 0) {
        sel_e[r][j] = bidx;
        sel_s[r][j] = best;
      }
    }
    __syncwarp();
    if (lane == 0) {
      float sum = sel_s[r][0];
      for (int j = 1; j < k; ++j) sum = __fadd_rn(sum, sel_s[r][j]);
      for (int j = 0; j < k; ++j) {
        topk_idx[r * k + j] = sel_e[r][j];
        topk_w[r * k + j] = __fdiv_rn(sel_s[r][j], sum);
      }
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
  if (tid == 0) {
    route->n_union = nu;
    hdr->router_arrivals = 0u;
  }
}

// ---------------------------------------------------------------------------------
// Weight streaming for K3 and K4. A CTA has 16 consumer warps and one producer warp; a
// ring of stages in shared memory is handed over with "full" and "empty" mbarriers, so
// the copies of the next stages are always in flight while the consumers compute. HBM
// serves long contiguous runs at full bandwidth and every copy operation has a fixed
// cost, so a stage is a few large copies of whole row segments of consecutive rows:
//  * boxed path (rows a multiple of 128 bytes, i.e. K a multiple of 256): the nibbles of
//    the stage's rows arrive as ONE TMA box per matrix over the view [128-byte chunk][row]
//    [128 bytes] with the 128-byte swizzle (granule j of row r stored at j ^ (r & 7), so
//    the MMA fragment reads are free of bank conflicts), and the fp16 scales as one 2D
//    TMA box per matrix;
//  * row path (other sizes): one 1D bulk copy per row segment into a row padded by 16
//    bytes, and the scales in 4-byte cp.async pieces.
// Work is assigned statically, so the split depends only on the sizes.
// ---------------------------------------------------------------------------------
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kMmaThreads = kConsumers + 32;            // + producer warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kChunkBlocks = 128;                       // Q4 blocks per row per stage (at most)
constexpr int kMaxRing = 4;
constexpr uint32_t kFullArrivals = 1 + 32;              // expect_tx + the producer's lanes
constexpr int kReducerWarps = 3;                         // gate/up: 16 rows x R <= 96 outputs
constexpr int kGuThreads = kMmaThreads + 32 * kReducerWarps;
constexpr int kConsumerBarrier = 1;                     // named barrier id of the consumers

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_addr(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__host__ __device__ constexpr size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// 1D bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-aligned).
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
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(kConsumers) : "memory");
}

// Row path: `rows` rows of `cb` blocks (nibbles and scales; row strides `row_qs` bytes /
// `nb` halves) into padded shared rows; called by all 32 producer lanes.
__device__ __forceinline__ void copy_rows(uint8_t* qdst, int qpitch, const uint8_t* qsrc,
                                          size_t row_qs, uint8_t* sdst, int spitch,
                                          const uint16_t* ssrc, int nb, int rows, int cb,
                                          uint64_t* bar, int lane) {
  for (int r = lane; r < rows; r += 32)
    bulk_copy(qdst + r * qpitch, qsrc + (size_t)r * row_qs, (uint32_t)cb * 16, bar);
  const int per_row = cb >> 1;
  for (int p = lane; p < rows * per_row; p += 32) {
    const int r = p / per_row, pp = p - r * per_row;
    cp_async4(sdst + r * spitch + pp * 4, ssrc + (size_t)r * nb + 2 * pp, true);
  }
}

// ---------------------------------------------------------------------------------
// K3: gate + up + SwiGLU. A unit is (expert slot u, 16 rows of I): slot 0 is the shared
// expert (all rows), slot u >= 1 the u-th expert of the union (its rows). CTA b takes
// units b, b + G, b + 2G, ... (G = grid). A stage is one K chunk of a unit (the gate and
// up rows' segments of up to 16 WB blocks); consumer warp w computes blocks WB w ..
// WB w + WB - 1 of the chunk for both matrices and keeps its partial sums across the
// unit's chunks. At the end of a unit the 16 warps' partials meet in shared memory and
// are added in warp order; h = bf16_rne(silu(g) * u) is written for the expert's rows.
// The activations sit in shared memory as bf16 in MMA pair order, staged once per CTA
// while the router runs. The producer starts on the shared expert's units before the
// router's results exist.
// ---------------------------------------------------------------------------------
// Stage geometry for WB blocks per warp (a chunk of 16 WB blocks per row): WB = 8 when
// the stages fit beside the staged activations, else 4.
template <int WB>
struct GuGeom {
  static constexpr int kCB = 16 * WB;                            // blocks per chunk
  static constexpr int kQsPitch = kCB * 16 + 16;                 // row path: 2064 / 1040
  static constexpr int kScPitch = kCB * 2 + 16;                  // row path: 272 / 144
  static constexpr int kRowQs = 2 * 16 * kQsPitch;               // row path: nibble bytes
  static constexpr int kBoxQs = 16 * kCB * 16;                   // boxed: one matrix
  static constexpr int kBoxSc = 16 * kCB * 2;                    // boxed: one matrix
  static constexpr int kStage = (int)round_up((size_t)kRowQs + 2 * 16 * kScPitch, 1024);
};
constexpr int kXPad = 64;                                  // staged activation row pad

struct alignas(64) GateUpArgs {
  CUtensorMap wq[4];   // boxed path: nibbles of gate, up, sh_gate, sh_up
  CUtensorMap wsc[4];  // boxed path: their scales
  Q4Ptr gate, up, sh_gate, sh_up;
  const uint16_t* x;
  const RouteInfo* route;
  uint16_t* h;
  uint32_t* status;
  int R, H, I, k, ring, boxed;
};

__host__ __device__ constexpr size_t gu_red_bytes(int R) {
  return 2ull * kConsumerWarps * 2 * 16 * (size_t)R * 4;
}

template <int WB>
__global__ void __launch_bounds__(kGuThreads, 1) k3_gate_up(const __grid_constant__ GateUpArgs a) {
  using Geo = GuGeom<WB>;
  // partial-sum buffers: written by the 16 consumer warps (pfull), read by the reducer
  // warps (pempty); two buffers, so consumers wait only when two units are unreduced
  __shared__ __align__(8) uint64_t s_pfull[2], s_pempty[2];
  constexpr int kCB = Geo::kCB, kStage = Geo::kStage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int R = a.R, H = a.H, I = a.I, k = a.k, ring = a.ring;
  const bool boxed = a.boxed != 0;
  const int nb = H >> 5;                          // Q4 blocks per row
  const int KC = (nb + kCB - 1) / kCB;
  const int RT = I >> 4;
  const int xstride = 2 * H + kXPad;
  const size_t row_qs = (size_t)H / 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;

  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)ring * kStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)ring * kStage + gu_red_bytes(R));
  uint64_t* empty = full + kMaxRing;
  uint8_t* xs = smem + (size_t)ring * kStage + gu_red_bytes(R) + 64;

  if (tid == 0) {
    for (int s = 0; s < ring; ++s) {
      mbar_init(&full[s], kFullArrivals);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_pfull[b], kConsumerWarps);
      mbar_init(&s_pempty[b], kReducerWarps);
    }
    fence_mbar_init();
    if (boxed)
      for (int i = 0; i < 4; ++i) { prefetch_tensormap(&a.wq[i]); prefetch_tensormap(&a.wsc[i]); }
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
    for (int f = 0;; ++f) {
      const int n = (int)blockIdx.x + (f / KC) * G, c = f % KC;
      const int u = n / RT, rti = n - u * RT;
      if (u > 0 && !routed) { pdl_wait(); routed = true; }
      if (routed && n >= (1 + a.route->n_union) * RT) break;
      const int slot = f % ring;
      if (f >= ring && !mbar_wait(&empty[slot], ((f / ring) - 1) & 1, kWaitPolls)) timed_out = true;
      uint8_t* st = stages + (size_t)slot * kStage;
      const int row0 = (u == 0 ? 0 : a.route->expert[u - 1] * I) + rti * 16;
      if (boxed) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], 2u * (Geo::kBoxQs + Geo::kBoxSc));
          const int mi = u == 0 ? 2 : 0;
          for (int m = 0; m < 2; ++m) {
            tma_load_3d(st + m * Geo::kBoxQs, &a.wq[mi + m], 0, row0, c * (kCB / 8), &full[slot]);
            tma_load_2d(st + 2 * Geo::kBoxQs + m * Geo::kBoxSc, &a.wsc[mi + m], c * kCB, row0,
                        &full[slot]);
          }
        }
      } else {
        const Q4Ptr mg = u == 0 ? a.sh_gate : a.gate, mu = u == 0 ? a.sh_up : a.up;
        const int cb = min(kCB, nb - c * kCB);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * 16u * cb * 16u);
        for (int m = 0; m < 2; ++m) {
          const Q4Ptr mm = m ? mu : mg;
          copy_rows(st + m * 16 * Geo::kQsPitch, Geo::kQsPitch,
                    mm.qs + (size_t)row0 * row_qs + (size_t)c * kCB * 16, row_qs,
                    st + Geo::kRowQs + m * 16 * Geo::kScPitch, Geo::kScPitch,
                    mm.sc + (size_t)row0 * nb + c * kCB, nb, 16, cb, &full[slot], lane);
        }
      }
      cp_async_mbar_arrive(&full[slot]);
    }
    if (!routed) pdl_wait();
  } else if (warp < kProducerWarp) {
    pdl_wait();      // the route produced by the router grid is visible from here on
    const RouteInfo* rt = a.route;
    const int n_units = (1 + rt->n_union) * RT;
    const int n_mine = (int)blockIdx.x < n_units ? (n_units - (int)blockIdx.x + G - 1) / G : 0;
    const int total = n_mine * KC;
    const uint8_t* xrow = xs + min(g, R - 1) * xstride + q * 16;   // rows >= R: any finite row
    // Byte offsets inside a stage (row g of the gate matrix; + m_q for up, + r8_q for row
    // g + 8) of word q of this warp's block j, and of this warp's scales.
    int woff[WB];
    int m_q, r8_q, soff, m_s, r8_s;
    if (boxed) {
#pragma unroll
      for (int j = 0; j < WB; ++j) {
        const int b = WB * warp + j;
        woff[j] = ((b >> 3) * 16 + g) * 128 + (((b & 7) ^ (g & 7)) << 4) + q * 4;
      }
      m_q = Geo::kBoxQs; r8_q = 8 * 128;
      soff = 2 * Geo::kBoxQs + g * (kCB * 2) + warp * (2 * WB);
      m_s = Geo::kBoxSc; r8_s = 8 * kCB * 2;
    } else {
#pragma unroll
      for (int j = 0; j < WB; ++j) woff[j] = g * Geo::kQsPitch + (WB * warp + j) * 16 + q * 4;
      m_q = 16 * Geo::kQsPitch; r8_q = 8 * Geo::kQsPitch;
      soff = Geo::kRowQs + g * Geo::kScPitch + warp * (2 * WB);
      m_s = 16 * Geo::kScPitch; r8_s = 8 * Geo::kScPitch;
    }
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    int buf = 0;
    for (int f = 0; f < total; ++f) {
      const int slot = f % ring;
      if (!mbar_wait(&full[slot], (f / ring) & 1, kWaitPolls)) timed_out = true;
      const uint8_t* st = stages + (size_t)slot * kStage;
      const int c = f % KC;
      const int cb = min(kCB, nb - c * kCB);
      const int nv = max(0, min(WB, cb - WB * warp));   // this warp's blocks in the chunk
      if (nv > 0) {
        // fp16 scales of rows g, g + 8 (gate, up) for the warp's WB blocks
        uint32_t sw[4][WB / 2];
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const uint8_t* p = st + soff + (m4 >> 1) * m_s + (m4 & 1) * r8_s;
          if constexpr (WB == 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(p);
            sw[m4][0] = v.x; sw[m4][1] = v.y; sw[m4][2] = v.z; sw[m4][3] = v.w;
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            sw[m4][0] = v.x; sw[m4][1] = v.y;
          }
        }
        const uint8_t* xb = xrow + (c * kCB + WB * warp) * 64;
#pragma unroll
        for (int jp = 0; jp < WB / 2; ++jp) {
          const float2 sg0 = __half22float2(*reinterpret_cast<const __half2*>(&sw[0][jp]));
          const float2 sg8 = __half22float2(*reinterpret_cast<const __half2*>(&sw[1][jp]));
          const float2 su0 = __half22float2(*reinterpret_cast<const __half2*>(&sw[2][jp]));
          const float2 su8 = __half22float2(*reinterpret_cast<const __half2*>(&sw[3][jp]));
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int j = 2 * jp + e2;
            if (j < nv) {
              const float g0 = e2 ? sg0.y : sg0.x, g8 = e2 ? sg8.y : sg8.x;
              const float u0 = e2 ? su0.y : su0.x, u8 = e2 ? su8.y : su8.x;
              const uint4 X = *reinterpret_cast<const uint4*>(xb + j * 64);
              const uint8_t* w = st + woff[j];
              float d[4];
              q4_block_mma(lds32(w), lds32(w + r8_q), X, d);
              ag[0] = __fmaf_rn(g0, d[0], ag[0]); ag[1] = __fmaf_rn(g0, d[1], ag[1]);
              ag[2] = __fmaf_rn(g8, d[2], ag[2]); ag[3] = __fmaf_rn(g8, d[3], ag[3]);
              q4_block_mma(lds32(w + m_q), lds32(w + m_q + r8_q), X, d);
              au[0] = __fmaf_rn(u0, d[0], au[0]); au[1] = __fmaf_rn(u0, d[1], au[1]);
              au[2] = __fmaf_rn(u8, d[2], au[2]); au[3] = __fmaf_rn(u8, d[3], au[3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);   // this warp is done with the slot
      if (c == KC - 1) {
        // partials [warp][gate/up][row][col] (cols < R only) into buffer unit & 1, once
        // the reducers are done with the unit that used it before
        const int unit = f / KC;
        if (unit >= 2 && !mbar_wait(&s_pempty[buf], ((unit >> 1) - 1) & 1, kWaitPolls))
          timed_out = true;
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
        buf ^= 1;
      }
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
      if (!mbar_wait(&s_pfull[b], (unit >> 1) & 1, kWaitPolls)) {
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
// K4: down projection. A unit is (expert slot u, a group of RS consecutive rows of H);
// the 16 consumer warps split a stage (one K chunk of up to 4096 values of the group's
// rows) into RS/16 row tiles x WK K slices of BPS blocks (16 where two stages fit, else 8;
// the larger slice halves the per-stage overhead per weight byte). CTA b takes a contiguous range of
// units, so consecutive stages mostly belong to one expert and its h (the B operand, kept
// in shared memory) is reloaded only when the expert or the chunk changes. The WK slice
// partials of a row tile are added in slice order and written to o[row][slot] (fp32);
// K5 combines. The weights do not depend on the gate/up kernel, so the producer starts
// streaming them before that kernel has finished; only h waits for it.
// ---------------------------------------------------------------------------------
struct DownGeom {
  int nb, KC, cbmax, WK, TPS, RS, NGR, qs_pitch, sc_pitch, h_pitch, stage_bytes, boxed;
};

__host__ __device__ inline DownGeom down_geom(int H, int I, int bps) {
  DownGeom d{};
  d.nb = I >> 5;
  d.KC = (d.nb + kChunkBlocks - 1) / kChunkBlocks;
  d.cbmax = d.nb < kChunkBlocks ? d.nb : kChunkBlocks;
  const int slices = (d.cbmax + bps - 1) / bps;
  d.WK = slices <= 1 ? 1 : (slices <= 2 ? 2 : (slices <= 4 ? 4 : (slices <= 8 ? 8 : 16)));
  d.TPS = kConsumerWarps / d.WK;
  d.RS = 16 * d.TPS;
  d.NGR = (H + d.RS - 1) / d.RS;
  d.boxed = (d.nb % 8) == 0;            // rows of whole 128-byte chunks (and scale rows of 16 B)
  d.qs_pitch = d.cbmax * 16 + 16;       // row path
  d.sc_pitch = (int)round_up((size_t)d.cbmax * 2, 16) + 16;
  d.h_pitch = d.cbmax * 64 + 64;
  d.stage_bytes = (int)round_up((size_t)d.RS * (d.qs_pitch + d.sc_pitch), 1024);
  return d;
}

struct alignas(64) DownArgs {
  CUtensorMap wq[2];   // boxed path: nibbles of down, sh_down
  CUtensorMap wsc[2];  // boxed path: their scales
  Q4Ptr down, sh_down;
  const uint16_t* h;
  const RouteInfo* route;
  float* opart;
  uint32_t* status;
  int R, H, I, k, ring, boxed;
};

__host__ __device__ constexpr size_t dn_red_bytes(int R) {
  return 2ull * kConsumerWarps * 16 * (size_t)R * 4;
}

template <int BPS>
__global__ void __launch_bounds__(kMmaThreads, 1) k4_down(const __grid_constant__ DownArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_rowmask[kMaxUnion];
  __shared__ __align__(8) int8_t s_slot[kMaxUnion][8];
  uint8_t* smem = align1024(smem_raw);
  const int R = a.R, H = a.H, I = a.I, k = a.k, ring = a.ring;
  const DownGeom dg = down_geom(H, I, BPS);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const size_t row_qs = (size_t)I / 2;

  uint8_t* stages = smem;
  uint8_t* hs = smem + (size_t)ring * dg.stage_bytes;                      // [8][h_pitch]
  float* red = reinterpret_cast<float*>(hs + (size_t)8 * dg.h_pitch);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(red) + dn_red_bytes(R));
  uint64_t* empty = full + kMaxRing;

  if (tid == 0) {
    for (int s = 0; s < ring; ++s) {
      mbar_init(&full[s], kFullArrivals);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
    if (a.boxed)
      for (int i = 0; i < 2; ++i) { prefetch_tensormap(&a.wq[i]); prefetch_tensormap(&a.wsc[i]); }
  }
  __syncthreads();

  // The route was complete before the gate/up kernel passed its own wait, which precedes
  // the launch of this grid; h is waited for below.
  const RouteInfo* rt = a.route;
  const int n_units = (1 + rt->n_union) * dg.NGR;
  const int G = gridDim.x;
  const int u_begin = (int)(((long long)blockIdx.x * n_units) / G);
  const int u_end = (int)(((long long)(blockIdx.x + 1) * n_units) / G);
  const int total = (u_end - u_begin) * dg.KC;
  const int box_qs = dg.RS * dg.cbmax * 16, box_sc = dg.RS * dg.cbmax * 2;
  bool timed_out = false;

  if (warp == kProducerWarp) {
    for (int f = 0; f < total; ++f) {
      const int slot = f % ring;
      if (f >= ring && !mbar_wait(&empty[slot], ((f / ring) - 1) & 1, kWaitPolls)) timed_out = true;
      uint8_t* st = stages + (size_t)slot * dg.stage_bytes;
      const int n = u_begin + f / dg.KC, c = f % dg.KC;
      const int u = n / dg.NGR, grp = n - u * dg.NGR;
      const int r0 = grp * dg.RS;
      const int row0 = (u == 0 ? 0 : rt->expert[u - 1] * H) + r0;
      if (a.boxed) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[slot], (uint32_t)(box_qs + box_sc));
          const int mi = u == 0 ? 1 : 0;
          tma_load_3d(st, &a.wq[mi], 0, row0, c * (kChunkBlocks / 8), &full[slot]);
          tma_load_2d(st + box_qs, &a.wsc[mi], c * kChunkBlocks, row0, &full[slot]);
        }
      } else {
        const Q4Ptr m = u == 0 ? a.sh_down : a.down;
        const int nrows = min(dg.RS, H - r0);
        const int cb = min(kChunkBlocks, dg.nb - c * kChunkBlocks);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)nrows * cb * 16u);
        copy_rows(st, dg.qs_pitch, m.qs + (size_t)row0 * row_qs + (size_t)c * kChunkBlocks * 16,
                  row_qs, st + dg.RS * dg.qs_pitch, dg.sc_pitch,
                  m.sc + (size_t)row0 * dg.nb + c * kChunkBlocks, dg.nb, nrows, cb, &full[slot],
                  lane);
      }
      cp_async_mbar_arrive(&full[slot]);
    }
    pdl_wait();
  } else {
    pdl_wait();      // h is complete from here on
    // the union's row masks and rank slots, read every stage, kept in shared memory
    for (int i = tid; i < rt->n_union; i += kConsumers) {
      s_rowmask[i] = rt->rowmask[i];
      *reinterpret_cast<uint2*>(s_slot[i]) = *reinterpret_cast<const uint2*>(rt->slot[i]);
    }
    consumer_sync();
    const int rtl = warp / dg.WK, ks = warp - rtl * dg.WK;   // row tile, K slice
    const int r = rtl * 16 + g;                              // this lane's first row
    // byte offset in a stage of word q of block j of this warp's slice (row r; + r8_q for
    // row r + 8), and of the slice's scales of row r (+ r8_s for row r + 8)
    auto woff = [&](int j) {
      const int b = ks * BPS + j;
      return a.boxed ? ((b >> 3) * dg.RS + r) * 128 + (((b & 7) ^ (r & 7)) << 4) + q * 4
                     : r * dg.qs_pitch + b * 16 + q * 4;
    };
    const int r8_q = a.boxed ? 8 * 128 : 8 * dg.qs_pitch;
    const int soff = a.boxed ? box_qs + r * (dg.cbmax * 2) + ks * (2 * BPS)
                             : dg.RS * dg.qs_pitch + r * dg.sc_pitch + ks * (2 * BPS);
    const int r8_s = a.boxed ? 8 * dg.cbmax * 2 : 8 * dg.sc_pitch;
    int h_tag = -1;     // (expert slot, chunk) whose h is staged
    int buf = 0;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int f = 0; f < total; ++f) {
      const int slot = f % ring;
      const int n = u_begin + f / dg.KC, c = f % dg.KC;
      const int u = n / dg.NGR, grp = n - u * dg.NGR;
      const int cb = min(kChunkBlocks, dg.nb - c * kChunkBlocks);
      const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : s_rowmask[u - 1];
      const int tag = u * dg.KC + c;
      if (tag != h_tag) {
        // h of the expert's rows for this chunk: [verify row][values], 16-byte pieces, then
        // each piece put in MMA pair order in place. Rows that do not use the expert keep
        // stale values; their MMA columns are never read.
        consumer_sync();   // every consumer is done with the previous h
        const int per_row = cb * 4;
        for (int p = tid; p < R * per_row; p += kConsumers) {
          const int rr = p / per_row, pp = p - rr * per_row;
          if ((rowmask >> rr) & 1u) {
            const int slot_r = (u == 0) ? 0 : s_slot[u - 1][rr];
            cp_async16(hs + rr * dg.h_pitch + pp * 16,
                       a.h + ((size_t)rr * (1 + k) + slot_r) * I + c * (kChunkBlocks * 32) + pp * 8,
                       true);
          }
        }
        cp_async_commit();
        cp_async_wait<0>();
        for (int p = tid; p < R * per_row; p += kConsumers) {
          const int rr = p / per_row, pp = p - rr * per_row;
          if ((rowmask >> rr) & 1u) {
            uint4* hp = reinterpret_cast<uint4*>(hs + rr * dg.h_pitch + pp * 16);
            *hp = pair_order(*hp);
          }
        }
        consumer_sync();
        h_tag = tag;
      }
      if (!mbar_wait(&full[slot], (f / ring) & 1, kWaitPolls)) timed_out = true;
      const uint8_t* st = stages + (size_t)slot * dg.stage_bytes;
      const int row_t = grp * dg.RS + rtl * 16;         // first row of this warp's tile
      const int nv = max(0, min(BPS, cb - BPS * ks));
      if (nv > 0 && row_t < H) {
        const uint8_t* hb = hs + g * dg.h_pitch + ks * (BPS * 64) + q * 16;
        // four blocks at a time: scales, activations and weights loaded before the MMAs
#pragma unroll
        for (int j0 = 0; j0 < BPS; j0 += 4) {
          if (j0 < nv) {
            float s0[4], s8[4];
            widen_scales(*reinterpret_cast<const uint2*>(st + soff + 2 * j0), s0);
            widen_scales(*reinterpret_cast<const uint2*>(st + soff + r8_s + 2 * j0), s8);
            uint4 X[4];
            uint32_t wl[4], wh[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              X[jj] = *reinterpret_cast<const uint4*>(hb + (j0 + jj) * 64);
              const uint8_t* w = st + woff(j0 + jj);
              wl[jj] = lds32(w);
              wh[jj] = lds32(w + r8_q);
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              if (j0 + jj < nv) {
                float d[4];
                q4_block_mma(wl[jj], wh[jj], X[jj], d);
                acc[0] = __fmaf_rn(s0[jj], d[0], acc[0]); acc[1] = __fmaf_rn(s0[jj], d[1], acc[1]);
                acc[2] = __fmaf_rn(s8[jj], d[2], acc[2]); acc[3] = __fmaf_rn(s8[jj], d[3], acc[3]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (c == dg.KC - 1) {
        // The WK slice warps of this row tile add their partials in slice order (a named
        // barrier per row tile, so the tiles do not wait for one another); with one slice
        // the warp writes its rows directly.
        if (dg.WK == 1) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = 2 * q + (e & 1), row = row_t + g + ((e & 2) ? 8 : 0);
            if (col < R && row < H && ((rowmask >> col) & 1u)) {
              const int slot_c = (u == 0) ? 0 : s_slot[u - 1][col];
              a.opart[((size_t)col * (1 + k) + slot_c) * H + row] = __fadd_rn(0.f, acc[e]);
            }
            acc[e] = 0.f;
          }
        } else {
          float* rb = red + (size_t)buf * kConsumerWarps * 16 * R;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = 2 * q + (e & 1), row = g + ((e & 2) ? 8 : 0);
            if (col < R) rb[(warp * 16 + row) * R + col] = acc[e];
            acc[e] = 0.f;
          }
          const int gthreads = dg.WK * 32, gt = tid - rtl * gthreads;
          asm volatile("bar.sync %0, %1;" ::"r"(2 + rtl), "r"(gthreads) : "memory");
          for (int t = gt; t < 16 * R; t += gthreads) {
            const int rr = t / R, col = t - rr * R;
            const int row = row_t + rr;
            if (row < H && ((rowmask >> col) & 1u)) {
              float o = 0.f;
              for (int s = 0; s < dg.WK; ++s)
                o = __fadd_rn(o, rb[((rtl * dg.WK + s) * 16 + rr) * R + col]);
              const int slot_c = (u == 0) ? 0 : s_slot[u - 1][col];
              a.opart[((size_t)col * (1 + k) + slot_c) * H + row] = o;
            }
          }
        }
        buf ^= 1;
      }
    }
  }
  pdl_trigger();
  if (timed_out && lane == 0) flag_status(a.status, kStatusTimeout);
}

// ---------------------------------------------------------------------------------
// K5: combine. y[r] = bf16_rne(o_shared + sum_j w_j o_j), the sum taken in rank order j.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k5_combine(const float* __restrict__ opart,
                                                  const float* __restrict__ topk_w,
                                                  uint16_t* __restrict__ y, int R, int H,
                                                  int k) {
  pdl_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= R * H) return;
  const int r = idx / H, col = idx - r * H;
  const float* o = opart + (size_t)r * (1 + k) * H + col;
  float yv = o[0];
  for (int j = 0; j < k; ++j) yv = __fmaf_rn(topk_w[r * k + j], o[(size_t)(1 + j) * H], yv);
  y[idx] = f32_to_bf16_rne(yv);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}


template <int WB>
size_t gate_up_smem(const MoeDims& d, int ring) {
  return 1024 + (size_t)ring * GuGeom<WB>::kStage + gu_red_bytes(d.R) + 64 +
         (size_t)d.R * (2 * d.H + kXPad);
}

size_t down_smem(const MoeDims& d, int ring, int bps) {
  const DownGeom g = down_geom(d.H, d.I, bps);
  return 1024 + (size_t)ring * g.stage_bytes + (size_t)8 * g.h_pitch + dn_red_bytes(d.R) + 64;
}

// Deepest ring (4 .. 2 stages) whose shared memory fits; 0 if none does.
template <typename F>
int pick_ring(F smem_of) {
  for (int ring = kMaxRing; ring >= 2; --ring)
    if (smem_of(ring) <= (size_t)device_max_smem_optin()) return ring;
  return 0;
}

template <int WB>
cudaError_t launch_gate_up_wb(const MoeDims& d, GateUpArgs& a, int ring, cudaStream_t s) {
  const size_t smem = gate_up_smem<WB>(d, ring);
  cudaError_t err = set_smem(k3_gate_up<WB>, smem);
  if (err != cudaSuccess) return err;
  a.ring = ring;
  if (a.boxed) {
    const Q4Ptr mats[4] = {a.gate, a.up, a.sh_gate, a.sh_up};
    for (int i = 0; i < 4; ++i) {
      const uint64_t rows = (uint64_t)(i < 2 ? d.E : 1) * d.I;
      if ((err = q4_maps(&a.wq[i], &a.wsc[i], mats[i], rows, d.H, 16, 16 * WB)) != cudaSuccess)
        return err;
    }
  }
  return launch_pdl(k3_gate_up<WB>, device_sm_count(), kGuThreads, smem, s, a);
}

}  // namespace

size_t gate_up_smem_bytes(const MoeDims& d) { return gate_up_smem<4>(d, 2); }

MoeLayout moe_layout(const MoeDims& d) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  MoeLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  L.zero_bytes = off;
  L.scores = off; off += up(sizeof(float) * (size_t)d.R * d.E);
  L.route = off; off += up(sizeof(RouteInfo));
  L.h = off; off += up(sizeof(uint16_t) * (size_t)d.R * (1 + d.k) * d.I);
  L.opart = off; off += up(sizeof(float) * (size_t)d.R * (1 + d.k) * d.H);
  L.total = off;
  return L;
}

cudaError_t launch_router(const MoeDims& d, const uint16_t* x, const uint16_t* router_w,
                          int32_t* topk_idx, float* topk_w, const MoeWorkspace& ws,
                          cudaStream_t s) {
  const int grid = (d.E + kRouterExperts - 1) / kRouterExperts;
  auto* hdr = reinterpret_cast<WsHeader*>(ws.header);
  if (d.E <= 12 * 32)
    k1_router<12><<<grid, kRouterWarps * 32, 0, s>>>(x, d.R, d.H, router_w, d.E, d.k, ws.scores,
                                                      topk_idx, topk_w, ws.route, hdr);
  else
    k1_router<kMaxExperts / 32><<<grid, kRouterWarps * 32, 0, s>>>(
        x, d.R, d.H, router_w, d.E, d.k, ws.scores, topk_idx, topk_w, ws.route, hdr);
  return cudaGetLastError();
}

cudaError_t launch_gate_up(const MoeDims& d, const uint16_t* x, Q4Ptr gate, Q4Ptr up,
                           Q4Ptr sh_gate, Q4Ptr sh_up, const MoeWorkspace& ws,
                           cudaStream_t s) {
  // Whole 4096-value chunks when they fit with a ring of at least 2, else half chunks.
  const int ring8 = pick_ring([&](int r) { return gate_up_smem<8>(d, r); });
  const int ring4 = pick_ring([&](int r) { return gate_up_smem<4>(d, r); });
  if (ring8 == 0 && ring4 == 0) return cudaErrorInvalidConfiguration;
  GateUpArgs a{};
  a.gate = gate; a.up = up; a.sh_gate = sh_gate; a.sh_up = sh_up;
  a.x = x; a.route = ws.route; a.h = ws.h; a.status = ws.header;
  a.R = d.R; a.H = d.H; a.I = d.I; a.k = d.k;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  a.boxed = (d.H % 256) == 0 && a16(gate.sc) && a16(up.sc) && a16(sh_gate.sc) && a16(sh_up.sc)
                ? 1 : 0;
  return ring8 ? launch_gate_up_wb<8>(d, a, ring8, s) : launch_gate_up_wb<4>(d, a, ring4, s);
}

cudaError_t launch_down(const MoeDims& d, Q4Ptr down, Q4Ptr sh_down, const float* topk_w,
                        uint16_t* y, const MoeWorkspace& ws, cudaStream_t s) {
  // 16 blocks per K slice where two stages fit (fewer stage overheads per byte), else 8
  int bps = 16;
  int ring = pick_ring([&](int r) { return down_smem(d, r, 16); });
  if (ring == 0) {
    bps = 8;
    ring = pick_ring([&](int r) { return down_smem(d, r, 8); });
  }
  if (ring == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = down_smem(d, ring, bps);
  auto kern = bps == 16 ? k4_down<16> : k4_down<8>;
  cudaError_t err = set_smem(kern, smem);
  if (err != cudaSuccess) return err;
  DownArgs a{};
  a.down = down; a.sh_down = sh_down; a.h = ws.h; a.route = ws.route; a.opart = ws.opart;
  a.status = ws.header;
  a.R = d.R; a.H = d.H; a.I = d.I; a.k = d.k; a.ring = ring;
  const DownGeom g = down_geom(d.H, d.I, bps);
  a.boxed = g.boxed && (reinterpret_cast<uintptr_t>(down.sc) & 15u) == 0 &&
            (reinterpret_cast<uintptr_t>(sh_down.sc) & 15u) == 0;
  if (a.boxed) {
    if ((err = q4_maps(&a.wq[0], &a.wsc[0], down, (uint64_t)d.E * d.H, d.I, g.RS, g.cbmax)) !=
            cudaSuccess ||
        (err = q4_maps(&a.wq[1], &a.wsc[1], sh_down, (uint64_t)d.H, d.I, g.RS, g.cbmax)) !=
            cudaSuccess)
      return err;
  }
  err = launch_pdl(kern, device_sm_count(), kMmaThreads, smem, s, a);
  if (err != cudaSuccess) return err;
  const int n = d.R * d.H;
  return launch_pdl(k5_combine, (n + 255) / 256, 256, 0, s, ws.opart, topk_w, y, d.R, d.H, d.k);
}

}  // namespace dsmoe
