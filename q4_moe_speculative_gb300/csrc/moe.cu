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
#include <algorithm>
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
// 1D bulk copy global -> shared of `bytes` (multiple of 16, both addresses 16-aligned),
// completing `bytes` of the transaction count of `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// The same with an L2 eviction-priority hint: the weights are read once per call, so they
// leave L2 first.
__device__ __forceinline__ void bulk_copy_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
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
// The layer as one persistent kernel, one CTA per SM, launched cooperatively so that every
// CTA is resident at once (the phases below wait on one another's results; every such
// wait is bounded and a give-up sets DS_ERR_TIMEOUT). Roles: 16 consumer warps, one
// producer warp, three reducer warps. Both weight phases stream through one ring of
// 36,864-byte stages in shared memory, handed over with "full" / "empty" mbarriers, so
// the producer moves on from the last gate/up stage to the first down stage at once.
//
//  1. Router. The consumers compute the sigmoid scores of experts b, b + G, ... (b = this
//     CTA, G = grid): thread t adds the products of chunks t, t + 512, ... of 8 values in
//     order, the lanes of a warp by a butterfly, the 16 warps in warp order. Once every
//     CTA has written its scores (an arrival count), every CTA reads them all and builds
//     the route itself: each row's top k (the largest key by a warp reduction per round,
//     ties to the lower expert), the renormalised weights, and the union of the selected
//     experts with each one's rows and rank slots, in shared memory. Meanwhile the
//     producer already streams the shared expert.
//  2. Gate + up + SwiGLU. A unit is (expert slot u, tile row of I = 16 rows): slot 0 is
//     the shared expert (all rows), slot u >= 1 the u-th expert of the union (its rows).
//     A stage is one K chunk of a unit: 32 tiles of the gate tile row and 32 of the up
//     tile row, two bulk copies. Consumer warp w takes tiles 2w, 2w + 1 of each chunk for
//     both matrices and keeps its partial sums across the unit's chunks; its activation
//     fragments for those tiles sit in tensor memory (written once, read back with
//     tcgen05.ld), which leaves shared memory to the ring. At the end of a unit the 16
//     warps' partials meet in shared memory; the reducer warps add them in warp order,
//     write h = bf16_rne(silu(g) * u) (each group of 8 values in MMA pair order) and count
//     the unit against its expert slot.
//  3. Down projection. A unit is (expert slot u, row group of 16 tile rows = 256 rows of
//     H); consumer warp w owns tile row w of the group for all of K (two accumulation
//     chains, even and odd tiles), so no reduction with other warps follows. A stage is 4
//     K tiles of the group's 16 tile rows, one contiguous bulk copy (the down matrices keep
//     their tile rows in groups of 16). The expert's h (the B operand) is brought into one
//     of two shared buffers by the producer, with bulk copies, once every gate/up unit of
//     the expert is counted. Each warp writes o[row][slot] (fp32).
//  Units are handed out by one atomic counter in a fixed order: every gate/up unit (the
//  shared expert's first), then every down unit, expert slot by expert slot. A CTA's
//  producer takes its next unit when the ring has room and records it with each stage, so
//  the CTAs stay busy until the last unit whatever their units' timing, and the gate/up
//  units of an expert are long done when its down units come up.
//  4. Combine. Once every CTA's down units are done (a count), CTA b writes y =
//     bf16_rne(o_shared + sum_j w_j o_j), j in rank order, for its share of H.
// ---------------------------------------------------------------------------------
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kReducerWarps = 3;                         // 16 rows x R <= 96 outputs
constexpr int kReducer0 = (kProducerWarp + 1) * 32;      // first reducer thread
constexpr int kMoeThreads = kReducer0 + 32 * kReducerWarps;
constexpr int kMaxRing = 8;
constexpr int kConsumerBarrier = 1;                      // named barrier: consumer warps
constexpr int kReducerBarrier = 2;                       // named barrier: reducer warps
constexpr int kXPad = 64;                                // staged h row pad (bytes)
constexpr int kGuCT = 32;                                // gate/up tiles per matrix per stage
constexpr int kDownKT = 4;                               // down tiles per tile row per stage
constexpr int kGroupRows = kDownGroup;                   // down tile rows per unit
constexpr int kStage = 2 * kGuCT * kTile;                // 36,864 bytes
static_assert(kGroupRows * kDownKT * kTile == kStage, "both phases share the stage size");
static_assert(kDownKT % 2 == 0, "down tiles alternate between two chains");
constexpr int kRouterBatch = 4;                          // experts per CTA per router batch

// Words of the workspace's zeroed area (the prologue clears it before every call): the
// status word, the router arrival count, the count of CTAs whose down outputs are written,
// the next unit to hand out, and from word kHdrUnits on, per expert slot, the gate/up units
// whose h is written.
enum : int { kHdrStatus = 0, kHdrArrivals = 1, kHdrDDone = 2, kHdrNext = 3, kHdrUnits = 64 };
constexpr int kMoeZeroBytes = 4 * (kHdrUnits + 128);
static_assert(kMaxUnion + 1 <= 128, "unit counts fit the zeroed area");

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded wait (about 1 s) until *p >= target; false on give-up.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t target) {
  for (uint32_t i = 0; i < (1u << 23); ++i) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(128);
  }
  return false;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_addr(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(kConsumers) : "memory");
}
__device__ __forceinline__ void reducer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kReducerBarrier), "n"(32 * kReducerWarps) : "memory");
}
// The reducer barrier, returning whether `pred` held in every reducer thread.
__device__ __forceinline__ bool reducer_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(kReducerBarrier), "n"(32 * kReducerWarps)
      : "memory");
  return r != 0;
}

struct MoeArgs {
  const uint16_t* x;          // bf16 [R][H]
  const uint16_t* router_w;   // bf16 [E][H]
  const uint8_t* gate;        // tiles [E][I/16][H/64], groups of 1
  const uint8_t* up;
  const uint8_t* down;        // tiles [E][H/16][I/64], groups of 16
  const uint8_t* sh_gate;
  const uint8_t* sh_up;
  const uint8_t* sh_down;
  float* scores;              // [R][E]
  RouteInfo* route;           // written by CTA 0 for inspection
  uint16_t* h;                // bf16 [R][1+k][I]
  float* opart;               // [R][1+k][H]
  int32_t* topk_idx;          // [R][k]
  float* topk_w;              // [R][k]
  uint16_t* y;                // bf16 [R][H]
  uint32_t* hdr;              // zeroed words (status, counts)
  int R, H, E, I, k, ring;
};

__host__ __device__ constexpr size_t moe_red_bytes(int R) {
  return (size_t)kConsumerWarps * 2 * 16 * R * 4;
}
// one staged h: the rows of one expert slot, rows of 2 I bytes + pad
__host__ __device__ constexpr size_t moe_h_bytes(int I, int R) { return (size_t)R * (2 * I + kXPad); }
// TMEM columns of the activation fragments: 16 per K chunk per warp, 4 warps per lane quarter.
__host__ __device__ constexpr uint32_t moe_tmem_cols(int H) {
  const int kc = (H / 64 + kGuCT - 1) / kGuCT;
  const uint32_t need = 64u * kc;
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

template <int KPER>   // score registers per lane in the top-k: ceil(E / 32) <= KPER
__global__ void __launch_bounds__(kMoeThreads, 1) k_moe(const MoeArgs a) {
  __shared__ __align__(8) uint64_t full[kMaxRing], empty[kMaxRing];
  // the partial sums of one gate/up unit: written by the 16 consumer warps (pfull), read by
  // the reducer warps (pempty); the route is built (s_route)
  __shared__ __align__(8) uint64_t s_pfull, s_pempty, s_route;
  // the two staged h buffers: filled by the producer (hfull), released by the consumers
  __shared__ __align__(8) uint64_t hfull[2], hempty[2];
  __shared__ int s_meta[kMaxRing];   // unit of each ring stage (-1: no unit left)
  __shared__ int s_red_unit[2];      // unit of the partials handed to the reducers (-1: end)
  __shared__ uint32_t s_tmem;
  __shared__ float s_part[kRouterBatch][kConsumerWarps][kMaxRows];
  __shared__ int32_t sel_e[kMaxRows][kMaxTopK];
  __shared__ float sel_s[kMaxRows][kMaxTopK];
  __shared__ uint32_t ubits[kMaxExperts / 32];
  __shared__ int16_t upos[kMaxExperts];
  __shared__ int32_t u_expert[kMaxUnion];
  __shared__ uint32_t u_rowmask[kMaxUnion];
  __shared__ __align__(8) int8_t u_slot[kMaxUnion][8];
  __shared__ int s_nunion;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int R = a.R, H = a.H, E = a.E, I = a.I, k = a.k, ring = a.ring;
  const int G = gridDim.x, b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  uint32_t* status = a.hdr + kHdrStatus;
  uint32_t* ucount = a.hdr + kHdrUnits;

  uint8_t* stages = smem;
  const size_t hbytes = moe_h_bytes(I, R);
  uint8_t* hbuf = smem + (size_t)ring * kStage;                    // [2][R][2 I + pad]
  float* red = reinterpret_cast<float*>(hbuf + 2 * hbytes);

  // gate/up geometry (K = H)
  const int Tg = H >> 6, KCg = (Tg + kGuCT - 1) / kGuCT, RTg = I >> 4;
  const size_t gu_expert = (size_t)RTg * Tg * kTile;
  // down geometry (K = I)
  const int Td = I >> 6, KCd = (Td + kDownKT - 1) / kDownKT, RTd = H >> 4;
  const int NGR = (RTd + kGroupRows - 1) / kGroupRows;
  const size_t dn_expert = (size_t)RTd * Td * kTile;
  const int hpitch = 2 * I + kXPad;
  const uint32_t tcols = moe_tmem_cols(H);

  if (tid == 0) {
    for (int s = 0; s < ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(&s_pfull, kConsumerWarps);
    mbar_init(&s_pempty, kReducerWarps);
    mbar_init(&s_route, 1);
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(&hfull[b2], 1);
      mbar_init(&hempty[b2], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool timed_out = false;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- producer ----------
    int slot = 0, f = 0;
    uint32_t phase = 0;    // ring cursor: stage f sits in `slot`, pass parity `phase`
    const uint64_t wpol = l2_evict_first();   // weights: read once per call
    int n_union = -1;      // known once this CTA has built the route
    auto routed = [&]() {
      if (n_union < 0) {
        if (!pipe_wait(&s_route, 0)) timed_out = true;
        n_union = s_nunion;
      }
    };
    auto next_slot = [&]() -> uint8_t* {
      if (f >= ring && !pipe_wait(&empty[slot], phase ^ 1u)) timed_out = true;
      return stages + (size_t)slot * kStage;
    };
    auto advance = [&]() {
      ++f;
      if (++slot == ring) { slot = 0; phase ^= 1u; }
    };
    // Units are handed out in one order to all CTAs (an atomic counter): every gate/up unit
    // (the shared expert's first: they need nothing from the router), then every down
    // unit, expert slot by expert slot. A CTA takes its next unit when its ring has room,
    // so the CTAs finish together whatever their units' timing; each stage records its
    // unit for the consumers, and after the last unit a stage carries the end marker.
    // The shared expert's unit b (b < S0 = min(G, RTg)) is taken first without the
    // counter: it needs neither the router nor the zeroed header, so it streams from the
    // start; the counter hands out the units from S0 on.
    const int S0 = min(G, RTg);
    int dn = 0;   // down units taken by this CTA (their h alternates between two buffers)
    bool own_first = b < S0, header_ready = false;
    for (;;) {
      int n = b;
      if (!own_first) {
        if (!header_ready) {
          pdl_wait();   // the prologue has zeroed the counter
          header_ready = true;
        }
        if (lane == 0) n = S0 + (int)atomicAdd(a.hdr + kHdrNext, 1u);
        n = __shfl_sync(0xffffffffu, n, 0);
      }
      own_first = false;
      if (n >= RTg) routed();
      const int NG = n_union >= 0 ? (1 + n_union) * RTg : RTg;
      const int ND = n_union >= 0 ? (1 + n_union) * NGR : 0;
      if (n >= NG + ND) {
        next_slot();
        if (lane == 0) {
          s_meta[slot] = -1;
          mbar_arrive(&full[slot]);
        }
        __syncwarp();
        break;
      }
      if (n < NG) {
        const int u = n / RTg, rt = n - u * RTg;
        const size_t e = u > 0 ? (size_t)u_expert[u - 1] : 0;
        const uint8_t* gb = u > 0 ? a.gate + e * gu_expert : a.sh_gate;
        const uint8_t* ub = u > 0 ? a.up + e * gu_expert : a.sh_up;
        for (int c = 0; c < KCg; ++c) {
          uint8_t* st = next_slot();
          if (lane == 0) {
            const size_t off = ((size_t)rt * Tg + (size_t)c * kGuCT) * kTile;
            const uint32_t bytes = (uint32_t)min(kGuCT, Tg - c * kGuCT) * kTile;
            s_meta[slot] = n;
            mbar_arrive_expect_tx(&full[slot], 2u * bytes);
            bulk_copy_hint(st, gb + off, bytes, &full[slot], wpol);
            bulk_copy_hint(st + kGuCT * kTile, ub + off, bytes, &full[slot], wpol);
          }
          __syncwarp();
          advance();
        }
      } else {
        const int m = n - NG, u = m / NGR, rg = m - u * NGR;
        const int hb = dn & 1;
        const int rig = min(kGroupRows, RTd - rg * kGroupRows);   // tile rows in the group
        const uint8_t* gbase = (u > 0 ? a.down + (size_t)u_expert[u - 1] * dn_expert : a.sh_down) +
                               (size_t)rg * kGroupRows * Td * kTile;
        auto issue = [&](int c) {
          uint8_t* st = next_slot();
          if (lane == 0) {
            const uint32_t bytes = (uint32_t)(min(kDownKT, Td - c * kDownKT) * rig * kTile);
            s_meta[slot] = n;
            mbar_arrive_expect_tx(&full[slot], bytes);
            bulk_copy_hint(st, gbase + (size_t)c * kDownKT * rig * kTile, bytes, &full[slot], wpol);
          }
          __syncwarp();
          advance();
        };
        // The unit's first `ring` stages need no h: their weights are on their way while
        // the expert's gate/up units finish (each takes a slot that an earlier unit's stage
        // frees, so none waits on this unit's h).
        const int pre = min(KCd, ring);
        for (int c = 0; c < pre; ++c) issue(c);
        if (lane == 0) {
          // h of the expert's rows, once every gate/up unit of the expert is counted and
          // the buffer's previous unit is done; h is stored in MMA pair order
          if (!wait_count(ucount + u, (uint32_t)RTg)) timed_out = true;
          if (dn >= 2 && !pipe_wait(&hempty[hb], ((dn >> 1) - 1) & 1)) timed_out = true;
          asm volatile("fence.proxy.async;" ::: "memory");   // h was written by other SMs
          const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : u_rowmask[u - 1];
          mbar_arrive_expect_tx(&hfull[hb], (uint32_t)__popc(rowmask) * 2u * (uint32_t)I);
          for (int rr = 0; rr < R; ++rr) {
            if ((rowmask >> rr) & 1u) {
              const int slot_r = (u == 0) ? 0 : u_slot[u - 1][rr];
              bulk_copy(hbuf + hb * hbytes + (size_t)rr * hpitch,
                        a.h + ((size_t)rr * (1 + k) + slot_r) * I, 2u * (uint32_t)I, &hfull[hb]);
            }
          }
        }
        __syncwarp();
        ++dn;
        for (int c = pre; c < KCd; ++c) issue(c);
      }
    }
  } else if (warp < kProducerWarp) {
    // ------------------------------------------------------------- consumers ---------
    // (1) router scores of experts b + j G
    for (int j0 = 0; b + j0 * G < E; j0 += kRouterBatch) {
      int ne = 0;
      while (ne < kRouterBatch && b + (j0 + ne) * G < E) ++ne;
      float acc[kRouterBatch][kMaxRows];
#pragma unroll
      for (int j = 0; j < kRouterBatch; ++j)
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) acc[j][r] = 0.0f;
      for (int ci = tid; ci < (H >> 3); ci += kConsumers) {
        uint4 wv[kRouterBatch], xv[kMaxRows];
#pragma unroll
        for (int j = 0; j < kRouterBatch; ++j)
          wv[j] = j < ne ? __ldcs(reinterpret_cast<const uint4*>(
                               a.router_w + (size_t)(b + (j0 + j) * G) * H + ci * 8))
                         : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
          xv[r] = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)min(r, R - 1) * H + ci * 8));
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          const uint32_t xw[4] = {xv[r].x, xv[r].y, xv[r].z, xv[r].w};
#pragma unroll
          for (int j = 0; j < kRouterBatch; ++j) {
            const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
            float t = acc[j][r];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              t = __fmaf_rn(bf16_lo(ww[m]), bf16_lo(xw[m]), t);
              t = __fmaf_rn(bf16_hi(ww[m]), bf16_hi(xw[m]), t);
            }
            acc[j][r] = t;   // rows >= R accumulate a copy of row R - 1, never read
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kRouterBatch; ++j)
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
          if (j < ne && r < R) {
            const float v = warp_sum(acc[j][r]);
            if (lane == 0) s_part[j][warp][r] = v;
          }
      consumer_sync();
      if (tid < ne * R) {
        const int j = tid / R, r = tid - j * R;
        float z = 0.0f;
        for (int w = 0; w < kConsumerWarps; ++w) z = __fadd_rn(z, s_part[j][w][r]);
        a.scores[r * E + b + (j0 + j) * G] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
      }
      consumer_sync();
    }
    // the prologue (zeroed header) is complete and visible from here on
    pdl_wait();
    // (2) every CTA's scores are written: count this one (the barrier orders its scores
    // before the fence), wait for all, then each CTA builds the route from all scores
    if (tid == 0) {
      __threadfence();
      atomicAdd(a.hdr + kHdrArrivals, 1u);
    }
    // While the other CTAs finish their scores: this warp's activation fragments -> tensor
    // memory. For each K chunk, tiles 2w and 2w + 1, each two blocks of 4 words in MMA pair
    // order (verify row g; rows >= R take a copy of row R - 1, any finite row): 16 columns
    // of this lane.
    const uint32_t tw = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(warp >> 2) * 16u * KCg;
    {
      const uint16_t* xg = a.x + (size_t)min(g, R - 1) * H + q * 8;
      for (int c = 0; c < KCg; ++c) {
        uint32_t v[16];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const int t = c * kGuCT + warp * 2 + tt;
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            uint4 w4 = make_uint4(0, 0, 0, 0);
            if (t < Tg) w4 = pair_order(__ldg(reinterpret_cast<const uint4*>(xg + (size_t)(2 * t + blk) * 32)));
            v[(tt * 2 + blk) * 4 + 0] = w4.x; v[(tt * 2 + blk) * 4 + 1] = w4.y;
            v[(tt * 2 + blk) * 4 + 2] = w4.z; v[(tt * 2 + blk) * 4 + 3] = w4.w;
          }
        }
        tmem_st16(tw + (uint32_t)c * 16u, v);
      }
    }
    if (tid == 0 && !wait_count(a.hdr + kHdrArrivals, (uint32_t)G)) timed_out = true;
    if (tid < kMaxExperts / 32) ubits[tid] = 0u;
    consumer_sync();
    if (warp < R) {
      // row r's top k by (score desc, expert asc): the warp-wide largest key, then the
      // smallest expert index holding it. Keys: score bits + 2 (sigmoid scores lie in
      // [0, 1]), 1 for NaN (from NaN inputs; below every score), 0 for none / taken.
      const int r = warp;
      uint32_t key[KPER];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < KPER; ++i) {
        const int e2 = i * 32 + lane;
        const float sv = e2 < E ? __ldcg(a.scores + r * E + e2) : 0.0f;
        bad |= (e2 < E) && !(sv >= 0.0f);
        key[i] = e2 >= E ? 0u : (sv >= 0.0f ? __float_as_uint(sv) + 2u : 1u);
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0 && b == 0) flag_status(status, kStatusCheck);
      for (int j = 0; j < k; ++j) {
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
      if (b == 0) {
        // renormalise: the sum in rank order (one lane), then one division per lane
        float sum = 0.0f;
        if (lane == 0) {
          sum = sel_s[r][0];
          for (int j = 1; j < k; ++j) sum = __fadd_rn(sum, sel_s[r][j]);
        }
        sum = __shfl_sync(0xffffffffu, sum, 0);
        if (lane < k) {
          a.topk_idx[r * k + lane] = sel_e[r][lane];
          a.topk_w[r * k + lane] = __fdiv_rn(sel_s[r][lane], sum);
        }
      }
    }
    consumer_sync();
    for (int i = tid; i < R * k; i += kConsumers) {
      const int e2 = sel_e[i / k][i % k];
      atomicOr(&ubits[e2 >> 5], 1u << (e2 & 31));
    }
    consumer_sync();
    if (warp == 0) {
      uint32_t bits = ubits[lane];
      const int c = __popc(bits);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nn = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nn;
      }
      int pos = incl - c;
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        const int e2 = lane * 32 + bit;
        upos[e2] = (int16_t)pos;
        u_expert[pos] = e2;
        u_rowmask[pos] = 0u;
        *reinterpret_cast<uint2*>(u_slot[pos]) = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        ++pos;
      }
      if (lane == 31) s_nunion = incl;
    }
    consumer_sync();
    for (int i = tid; i < R * k; i += kConsumers) {
      const int r = i / k, j = i % k;
      const int p = upos[sel_e[r][j]];
      atomicOr(&u_rowmask[p], 1u << r);
      u_slot[p][r] = (int8_t)(j + 1);
    }
    consumer_sync();
    const int n_union = s_nunion;
    if (tid == 0) mbar_arrive(&s_route);   // the producer and the reducers may read it now
    if (b == 0) {   // a copy of the route for inspection
      for (int i = tid; i < n_union; i += kConsumers) {
        a.route->expert[i] = u_expert[i];
        a.route->rowmask[i] = u_rowmask[i];
        *reinterpret_cast<uint2*>(a.route->slot[i]) = *reinterpret_cast<const uint2*>(u_slot[i]);
      }
      if (tid == 0) a.route->n_union = n_union;
    }
    // (3) / (4) the units the producer took, in its order
    const int NG = (1 + n_union) * RTg;
    const uint8_t* const hrow0 = hbuf + (size_t)min(g, R - 1) * hpitch + q * 16;   // rows >= R: a copy
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    // down: two chains, even (acc) and odd (acc2) tiles of the row, added at the unit end
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    int slot = 0;
    uint32_t phase = 0;
    int gu_k = 0;   // gate/up units handed to the reducers
    int dn = 0;     // down units done
    for (;;) {
      if (!pipe_wait(&full[slot], phase)) { timed_out = true; break; }
      const int n = s_meta[slot];
      if (n < 0) break;
      if (n < NG) {
        // gate/up: KCg stages; warp w takes tiles 2w, 2w + 1 of each
        for (int c = 0; c < KCg; ++c) {
          if (c > 0 && !pipe_wait(&full[slot], phase)) timed_out = true;
          const uint8_t* st = stages + (size_t)slot * kStage;
          const int ct = min(kGuCT, Tg - c * kGuCT);
#pragma unroll
          for (int tt = 0; tt < 2; ++tt) {
            const int t = warp * 2 + tt;
            if (t < ct) {
              uint32_t xw[8];   // blocks 2t, 2t + 1 of the chunk
              tmem_ld8(tw + (uint32_t)(c * 16 + tt * 8), xw);
              const uint4 X0 = make_uint4(xw[0], xw[1], xw[2], xw[3]);
              const uint4 X1 = make_uint4(xw[4], xw[5], xw[6], xw[7]);
              const uint8_t* tg = st + t * kTile;
              const uint8_t* tu = st + (kGuCT + t) * kTile;
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
        // partials [warp][gate/up][row][col] (cols < R only), once the reducers are done
        // with the unit before
        if (gu_k >= 1 && !pipe_wait(&s_pempty, (gu_k - 1) & 1)) timed_out = true;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = 2 * q + (e & 1), row = g + ((e & 2) ? 8 : 0);
          if (col < R) {
            red[((warp * 2 + 0) * 16 + row) * R + col] = ag[e];
            red[((warp * 2 + 1) * 16 + row) * R + col] = au[e];
          }
          ag[e] = 0.f;
          au[e] = 0.f;
        }
        if (tid == 0) s_red_unit[gu_k & 1] = n;
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_pfull);
        ++gu_k;
      } else {
        // down: warp w owns tile row w of the group for all of K
        const int m = n - NG, u = m / NGR, rg = m - u * NGR;
        const int rig = min(kGroupRows, RTd - rg * kGroupRows);
        const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : u_rowmask[u - 1];
        const int hb = dn & 1;
        if (!pipe_wait(&hfull[hb], (dn >> 1) & 1)) timed_out = true;
        const uint8_t* hrow = hrow0 + hb * hbytes;
        const int tr = rg * kGroupRows + warp;              // this warp's tile row
        for (int c = 0; c < KCd; ++c) {
          if (c > 0 && !pipe_wait(&full[slot], phase)) timed_out = true;
          const uint8_t* st = stages + (size_t)slot * kStage;
          const int kt = min(kDownKT, Td - c * kDownKT);
          if (warp < rig) {
            const uint8_t* xc = hrow + (size_t)c * kDownKT * 128;
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&hempty[hb]);   // this warp is done with the staged h
        ++dn;
        if (warp < rig) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = 2 * q + (e & 1), row = tr * 16 + g + ((e & 2) ? 8 : 0);
            if (col < R && ((rowmask >> col) & 1u)) {
              const int slot_c = (u == 0) ? 0 : u_slot[u - 1][col];
              a.opart[((size_t)col * (1 + k) + slot_c) * H + row] = __fadd_rn(acc[e], acc2[e]);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = acc2[e] = 0.f;
      }
    }
    tc_fence_before();   // this warp's tensor-memory reads are done
    // the reducers stop at an end marker in place of a unit. It is handed over only once
    // they are done with the last unit, as every unit is: a waiter on a parity must not
    // see two phases complete while it looks away.
    if (gu_k >= 1 && !pipe_wait(&s_pempty, (gu_k - 1) & 1)) timed_out = true;
    if (tid == 0) s_red_unit[gu_k & 1] = -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_pfull);
    // this CTA's outputs are written: count it (the barrier orders them before the fence)
    consumer_sync();
    if (tid == 0) {
      __threadfence();
      atomicAdd(a.hdr + kHdrDDone, 1u);
    }
  } else {
    // ------------------------------------------------------------- reducers ----------
    // For each gate/up unit of this CTA, in order, the 16 warps' partials are added in warp
    // order, h = bf16_rne(silu(g) * u) is written for the expert's rows, and the unit is
    // counted against its expert slot.
    const int rtid = tid - kReducer0;
    pdl_wait();   // the prologue (zeroed header) is complete
    if (!pipe_wait(&s_route, 0)) timed_out = true;
    for (int unit = 0;; ++unit) {
      // the three warps leave together on a give-up (they meet at a named barrier below)
      if (!reducer_all(pipe_wait(&s_pfull, unit & 1))) { timed_out = true; break; }
      const int n = s_red_unit[unit & 1];
      if (n < 0) break;
      const int u = n / RTg, rti = n - u * RTg;
      if (rtid < 16 * R) {
        const int row = rtid / R, col = rtid - row * R;
        const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : u_rowmask[u - 1];
        if ((rowmask >> col) & 1u) {
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) {
            gs = __fadd_rn(gs, red[((w * 2 + 0) * 16 + row) * R + col]);
            us = __fadd_rn(us, red[((w * 2 + 1) * 16 + row) * R + col]);
          }
          const int slot_c = (u == 0) ? 0 : u_slot[u - 1][col];
          const float silu = __fdiv_rn(gs, __fadd_rn(1.0f, expf(-gs)));
          // value i = rti * 16 + row, stored in MMA pair order within its group of 8
          // (v0, v4, v1, v5, v2, v6, v3, v7)
          const int i = rti * 16 + row, i8 = i & 7;
          const int pos = (i & ~7) | (i8 < 4 ? 2 * i8 : 2 * (i8 - 4) + 1);
          a.h[((size_t)col * (1 + k) + slot_c) * I + pos] = f32_to_bf16_rne(__fmul_rn(silu, us));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_pempty);
      // the unit's h is written by all three warps: count it (the barrier orders the
      // writes before the fence)
      reducer_sync();
      if (rtid == 0) {
        __threadfence();
        atomicAdd(ucount + u, 1u);
      }
    }
  }

  // (5) combine, once every CTA's down outputs are written: rows [H b / G, H (b+1) / G)
  if (tid == 0 && !wait_count(a.hdr + kHdrDDone, (uint32_t)G)) timed_out = true;
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
  const int r0 = (int)(((long long)b * H) / G), r1 = (int)(((long long)(b + 1) * H) / G);
  const int nrows = r1 - r0;
  for (int i = tid; i < R * nrows; i += kMoeThreads) {
    const int r = i / nrows, row = r0 + (i - r * nrows);
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
  if (timed_out && lane == 0) flag_status(status, kStatusTimeout);
}

size_t moe_smem(const MoeDims& d, int ring) {
  return 1024 + (size_t)ring * kStage + 2 * moe_h_bytes(d.I, d.R) + moe_red_bytes(d.R);
}

// Deepest ring (kMaxRing .. 2 stages) whose shared memory fits beside the kernel's static
// shared memory (under 8 KB); 0 if none does.
int moe_ring(const MoeDims& d) {
  for (int ring = kMaxRing; ring >= 2; --ring)
    if (moe_smem(d, ring) + 8 * 1024 <= (size_t)device_max_smem_optin()) return ring;
  return 0;
}

template <int KPER>
cudaError_t launch_moe_k(const MoeArgs& a, size_t smem, cudaStream_t s) {
  // the shared-memory attribute and the one-CTA-per-SM check, once per device and size
  static thread_local int set_dev = -1;
  static thread_local size_t set_smem = 0;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev != set_dev || smem != set_smem) {
    err = cudaFuncSetAttribute(k_moe<KPER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_moe<KPER>, kMoeThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    set_dev = dev;
    set_smem = smem;
  }
  // one CTA per SM, all resident at once (cooperative launch), allowed to start while the
  // prologue before it finishes (programmatic dependent launch: the kernel waits for the
  // prologue before it touches the workspace header)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(device_sm_count());
  cfg.blockDim = dim3(kMoeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_moe<KPER>, a);
}

}  // namespace

bool moe_fits(const MoeDims& d) { return moe_ring(d) != 0; }

MoeLayout moe_layout(const MoeDims& d) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  MoeLayout L{};
  size_t off = 0;
  L.header = off; off += kMoeZeroBytes;
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

cudaError_t launch_moe(const MoeDims& d, const uint16_t* x, const uint16_t* router_w,
                       const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                       const uint8_t* sh_gate, const uint8_t* sh_up, const uint8_t* sh_down,
                       int32_t* topk_idx, float* topk_w, uint16_t* y, const MoeWorkspace& ws,
                       cudaStream_t s, cudaEvent_t after_prologue) {
  // zero the header (status, arrival counts, flags): a plain launch, after the stream's
  // earlier work
  k0_clear<<<1, 256, 0, s>>>(ws.header, (int)(ws.zero_bytes / 4));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (after_prologue && (err = cudaEventRecord(after_prologue, s)) != cudaSuccess) return err;
  const int ring = moe_ring(d);
  if (ring == 0) return cudaErrorInvalidConfiguration;
  MoeArgs a{};
  a.x = x; a.router_w = router_w;
  a.gate = gate; a.up = up; a.down = down; a.sh_gate = sh_gate; a.sh_up = sh_up; a.sh_down = sh_down;
  a.scores = ws.scores; a.route = ws.route; a.h = ws.h; a.opart = ws.opart;
  a.topk_idx = topk_idx; a.topk_w = topk_w; a.y = y; a.hdr = ws.header;
  a.R = d.R; a.H = d.H; a.E = d.E; a.I = d.I; a.k = d.k; a.ring = ring;
  const size_t smem = moe_smem(d, ring);
  if (d.E <= 12 * 32) return launch_moe_k<12>(a, smem, s);
  return launch_moe_k<kMaxExperts / 32>(a, smem, s);
}

}  // namespace dsmoe
