// q8.cu — paired Q8 projections: R verify rows (R <= 8) through one Q8 weight matrix, every
// weight byte loaded from HBM once and applied to all rows.
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)", paragraph
// "DSpark": the 6 verify rows share one weight stream through paired Q8 projections.
//
// Format: blocks of 32 int8 values (two's complement) along K with one fp16 scale per
// block, value = scale * q. The kernels stream the tile-major form written once by
// k0_q8_tile: a tile is 16 rows x 64 values (two blocks) in 1088 bytes, 1024 bytes of int8
// in tensor-core fragment order followed by 64 bytes of scales. For block j of a tile,
// lane L = 4g + q holds at 512 j + 16 L the bytes k = 4q .. 4q+3 of rows g and g + 8 for the
// block's first 16 values, then the same for its last 16 values; the scales of lane group g
// sit at 1024 + 8 g as (row g block 0, row g+8 block 0, row g block 1, row g+8 block 1).
// Tiles run along K within a 16-row unit and units follow one another, so a matrix is one
// contiguous stream.
//
// Dot products run as mma.sync m16n8k16 (bf16 in, fp32 accumulate): a 32-bit word of four
// int8 values becomes two bf16 pairs with a shift, four AND-ORs and two bf16x2
// subtractions, exactly: (w & 0x007F007F) | 0x43004300 is (128 + low 7 bits) per half, the
// sign bit selects 128 or 256 to subtract. Within each 16-value step the K order is
// (4q, 4q+2 | 4q+1, 4q+3) for lane q, a permutation shared by the weights and the
// activations. Each block's scale multiplies its two MMAs' fp32 result once.
//
// k_q8_proj: one CTA per SM over a contiguous range of 16-row units; a producer warp moves
// stages of 16 consecutive tiles (17 KB) with 1D bulk copies into a ring; consumer warp w
// takes tile w of every stage (so K tiles w, w + 16, ... of every unit) and keeps one fp32
// partial per unit; the 16 partials of a unit are added in warp order by the warp that
// completes the unit, and rounded once to bf16. Nothing depends on R or on the other rows, so an R-row
// call writes the same bytes as R one-row calls.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace dsmoe {
namespace {

using namespace sm100;

constexpr int kWarps = 16;                       // consumer warps
constexpr int kThreads = 32 * (kWarps + 1);      // + one producer warp
constexpr int kStageTiles = kWarps;              // one tile per consumer warp per stage
constexpr int kStageBytes = kStageTiles * kQ8TileBytes;
constexpr uint32_t kWaitSleepNs = 2000;
constexpr uint32_t kWaitPolls = (1u << 30) / kWaitSleepNs;   // about 1 s in all

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
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
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_sleep(bar, parity, kWaitPolls, kWaitSleepNs);
}

// The int8 values at bytes 0 and 2 of w as a bf16 pair, exactly.
__device__ __forceinline__ uint32_t q8_pair(uint32_t w) {
  uint32_t m, c, d;
  asm("lop3.b32 %0, %1, 0x007F007F, 0x43004300, 0xEA;" : "=r"(m) : "r"(w));
  asm("lop3.b32 %0, %1, 0x00800080, 0x43004300, 0xEA;" : "=r"(c) : "r"(w));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(m), "r"(c));
  return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// One Q8 block for the 16 rows of a tile: W holds this lane's words (row g step 0, row g+8
// step 0, row g step 1, row g+8 step 1), X the matching activation pairs of verify row g.
// Returns the raw block dot products D[row g / g+8][col 2q, 2q+1].
__device__ __forceinline__ void q8_block_mma(const uint4& W, const uint4& X, float (&d)[4]) {
  const float z[4] = {0.f, 0.f, 0.f, 0.f};
  mma16816(d, q8_pair(W.x), q8_pair(W.y), q8_pair(W.x >> 8), q8_pair(W.y >> 8), X.x, X.y, z);
  mma16816(d, q8_pair(W.z), q8_pair(W.w), q8_pair(W.z >> 8), q8_pair(W.w >> 8), X.z, X.w, d);
}

struct Q8Args {
  const uint8_t* tiles;   // tile-major Q8 [rows/16][K/64] tiles
  int rows, K, R;
  const uint16_t* x;      // bf16 [R][K]
  uint16_t* y;            // bf16 [R][rows]
  uint32_t* status;
  int stages, slots;      // ring depth, partial slots
};

__host__ __device__ inline size_t q8_xs_bytes(int R, int K) { return (size_t)2 * R * K; }
__host__ __device__ inline size_t q8_slot_bytes() { return (size_t)kWarps * 32 * 16; }

// ---------------------------------------------------------------------------------
// k0_q8_tile: planar Q8 (qs int8 [rows][K], sc fp16 [rows][K/32]) -> tile-major. One
// thread per (tile, lane).
// ---------------------------------------------------------------------------------
__global__ void k0_q8_tile(const int8_t* qs, const uint16_t* sc, int rows, int K,
                           uint8_t* dst) {
  const int Tk = K / 64;
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long ntile = (long long)(rows / 16) * Tk;
  if (t >= ntile * 32) return;
  const long long tile = t >> 5;
  const int L = (int)(t & 31), g = L >> 2, q = L & 3;
  const int u = (int)(tile / Tk), kt = (int)(tile - (long long)u * Tk);
  const int r0 = 16 * u + g, r1 = r0 + 8;
  uint8_t* out = dst + tile * kQ8TileBytes;
  for (int j = 0; j < 2; ++j) {
    const int kb = 64 * kt + 32 * j;
    uint32_t w[4];
    const int ks[4] = {kb + 4 * q, kb + 4 * q, kb + 16 + 4 * q, kb + 16 + 4 * q};
    const int rs[4] = {r0, r1, r0, r1};
    for (int e = 0; e < 4; ++e)
      w[e] = *reinterpret_cast<const uint32_t*>(qs + (size_t)rs[e] * K + ks[e]);
    *reinterpret_cast<uint4*>(out + 512 * j + 16 * L) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (q == 0) {
    const size_t S = (size_t)K / 32;
    const uint16_t s4[4] = {sc[r0 * S + 2 * kt], sc[r1 * S + 2 * kt], sc[r0 * S + 2 * kt + 1],
                            sc[r1 * S + 2 * kt + 1]};
    *reinterpret_cast<uint2*>(out + 1024 + 8 * g) =
        make_uint2(s4[0] | ((uint32_t)s4[1] << 16), s4[2] | ((uint32_t)s4[3] << 16));
  }
}

// ---------------------------------------------------------------------------------
// k_q8_proj (layout of the dynamic shared memory: activations, partial slots, ring).
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) k_q8_proj(const __grid_constant__ Q8Args a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_full[kQ8MaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kQ8MaxStages];
  __shared__ int s_cnt[kQ8MaxSlots];
  __shared__ volatile int s_abort;
  const int S = a.stages, P = a.slots;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Tk = a.K / 64, units = a.rows / 16;
  const int u0 = (int)(((long long)blockIdx.x * units) / gridDim.x);
  const int u1 = (int)(((long long)(blockIdx.x + 1) * units) / gridDim.x);
  const int nstage = (u1 - u0) * Tk / kStageTiles;   // Tk is a multiple of kStageTiles
  uint4* xs = reinterpret_cast<uint4*>(smem);        // [K/32 blocks][R][4 q] activation pairs
  float4* slot = reinterpret_cast<float4*>(smem + q8_xs_bytes(a.R, a.K));  // [P][warps][32]
  uint8_t* ring = smem + q8_xs_bytes(a.R, a.K) + (size_t)P * q8_slot_bytes();

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < P; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  pdl_trigger();   // the next grid may start launching (it waits for this one's outputs)
  if (warp == kWarps) {
    // The weights do not come from the grid before this one (a programmatic launch): the
    // ring fills while it finishes.
    // ------------------------------------------------------------- producer ------
    if (lane == 0) {
      const uint8_t* src = a.tiles + (size_t)u0 * Tk * kQ8TileBytes;
      int s = 0;
      uint32_t par = 1;   // parity of the empty phase to wait for (from the second lap on)
      for (int i = 0; i < nstage; ++i) {
        if (i >= S && (s_abort || !pipe_wait(&bar_empty[s], par))) {
          s_abort = 1;
          flag_status(a.status, kStatusTimeout);
          break;
        }
        mbar_arrive_expect_tx(&bar_full[s], kStageBytes);
        bulk_copy(ring + (size_t)s * kStageBytes, src + (size_t)i * kStageBytes, kStageBytes,
                  &bar_full[s]);
        if (++s == S) {
          s = 0;
          par ^= 1u;
        }
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers -------
  // The activations may come from the grid before this one: wait for it. The call's
  // status word is reset here (a give-up is flagged only after a wait of about 1 s).
  pdl_wait();
  if (blockIdx.x == 0 && tid == 0) *a.status = 0u;
  // activations of verify row g, block b, lane q: (x[4q], x[4q+2]), (x[4q+1], x[4q+3]) of
  // the block's first 16 values, then the same for its last 16 (bf16 pairs); staged by the
  // consumer warps while the producer starts the weight stream
  {
    const int n = (a.K / 32) * a.R * 4;
#pragma unroll 4
    for (int i = tid; i < n; i += 32 * kWarps) {
      const int q = i & 3, g = (i >> 2) % a.R, b = (i >> 2) / a.R;
      const uint16_t* xr = a.x + (size_t)g * a.K + 32 * b + 4 * q;
      const uint2 lo = __ldg(reinterpret_cast<const uint2*>(xr));        // 4q .. 4q+3
      const uint2 hi = __ldg(reinterpret_cast<const uint2*>(xr + 16));   // 16+4q .. 16+4q+3
      uint4 v;
      v.x = __byte_perm(lo.x, lo.y, 0x5410);   // (x0, x2)
      v.y = __byte_perm(lo.x, lo.y, 0x7632);   // (x1, x3)
      v.z = __byte_perm(hi.x, hi.y, 0x5410);
      v.w = __byte_perm(hi.x, hi.y, 0x7632);
      xs[i] = v;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kWarps) : "memory");
  }
  const int g = lane >> 2, q = lane & 3;
  const bool xrow = g < a.R;
  const int per_unit = Tk / kStageTiles;   // stages per unit
  // this warp's activation fragments: K tile kt = upos * kStageTiles + warp of the unit,
  // blocks 2 kt and 2 kt + 1 at xs[8 R kt + 4 g + q] and 4 R further
  const int x_first = 8 * a.R * warp + 4 * g + q, x_step = 8 * a.R * kStageTiles;
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  int s = 0, upos = 0, sl = 0, u = u0, xo = x_first;
  uint32_t par = 0;
  for (int i = 0; i < nstage; ++i) {
    if (s_abort || !pipe_wait(&bar_full[s], par)) {
      if (lane == 0) {
        s_abort = 1;
        flag_status(a.status, kStatusTimeout);
      }
      break;
    }
    const uint8_t* tile = ring + (size_t)s * kStageBytes + (size_t)warp * kQ8TileBytes;
    const uint4 W0 = *reinterpret_cast<const uint4*>(tile + 16 * lane);
    const uint4 W1 = *reinterpret_cast<const uint4*>(tile + 512 + 16 * lane);
    const uint2 sc = *reinterpret_cast<const uint2*>(tile + 1024 + 8 * g);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_empty[s]);   // this warp's tile is in registers
    if (++s == S) {
      s = 0;
      par ^= 1u;
    }
    const uint4 X0 = xrow ? xs[xo] : zero4;
    const uint4 X1 = xrow ? xs[xo + 4 * a.R] : zero4;
    xo += x_step;
    float d[4];
    q8_block_mma(W0, X0, d);
    {
      const float s_g = __half2float(__ushort_as_half((unsigned short)(sc.x & 0xFFFF)));
      const float s_g8 = __half2float(__ushort_as_half((unsigned short)(sc.x >> 16)));
      acc[0] = __fmaf_rn(s_g, d[0], acc[0]);
      acc[1] = __fmaf_rn(s_g, d[1], acc[1]);
      acc[2] = __fmaf_rn(s_g8, d[2], acc[2]);
      acc[3] = __fmaf_rn(s_g8, d[3], acc[3]);
    }
    q8_block_mma(W1, X1, d);
    {
      const float s_g = __half2float(__ushort_as_half((unsigned short)(sc.y & 0xFFFF)));
      const float s_g8 = __half2float(__ushort_as_half((unsigned short)(sc.y >> 16)));
      acc[0] = __fmaf_rn(s_g, d[0], acc[0]);
      acc[1] = __fmaf_rn(s_g, d[1], acc[1]);
      acc[2] = __fmaf_rn(s_g8, d[2], acc[2]);
      acc[3] = __fmaf_rn(s_g8, d[3], acc[3]);
    }
    if (++upos != per_unit) continue;
    // the unit is complete for this warp: its partial into the unit's slot; the warp that
    // completes the unit adds the partials in warp order and writes y
    upos = 0;
    xo = x_first;
    const int uu = u, ss = sl;
    ++u;
    if (++sl == P) sl = 0;
    slot[((size_t)ss * kWarps + warp) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    __threadfence_block();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&s_cnt[ss], 1) == kWarps - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __threadfence_block();
    float4 t = slot[((size_t)ss * kWarps) * 32 + lane];
    for (int w = 1; w < kWarps; ++w) {
      const float4 v = slot[((size_t)ss * kWarps + w) * 32 + lane];
      t.x = __fadd_rn(t.x, v.x);
      t.y = __fadd_rn(t.y, v.y);
      t.z = __fadd_rn(t.z, v.z);
      t.w = __fadd_rn(t.w, v.w);
    }
    __syncwarp();
    if (lane == 0) s_cnt[ss] = 0;   // the slot is free for unit uu + P
    const int row = 16 * uu + g, c0 = 2 * q, c1 = 2 * q + 1;
    if (c0 < a.R) {
      a.y[(size_t)c0 * a.rows + row] = __bfloat16_as_ushort(__float2bfloat16_rn(t.x));
      a.y[(size_t)c0 * a.rows + row + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(t.z));
    }
    if (c1 < a.R) {
      a.y[(size_t)c1 * a.rows + row] = __bfloat16_as_ushort(__float2bfloat16_rn(t.y));
      a.y[(size_t)c1 * a.rows + row + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(t.w));
    }
  }
}

}  // namespace

size_t q8_tiled_bytes(long long rows, int K) {
  return (size_t)(rows / 16) * (size_t)(K / 64) * kQ8TileBytes;
}

cudaError_t launch_q8_tile(const int8_t* qs, const uint16_t* sc, int rows, int K, void* dst,
                           cudaStream_t s) {
  const long long threads = (long long)(rows / 16) * (K / 64) * 32;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  k0_q8_tile<<<(unsigned)grid, block, 0, s>>>(qs, sc, rows, K, static_cast<uint8_t*>(dst));
  return cudaGetLastError();
}

// Ring depth and partial slots for an R x K call, or false when the activations leave no
// room for a useful ring (at least 4 stages).
bool q8_plan(int R, int K, int* stages, int* slots, size_t* smem) {
  const size_t budget = (size_t)device_max_smem_optin() - 2048;
  const size_t xs = q8_xs_bytes(R, K);
  const int Tk = K / 64, per_unit = Tk / kStageTiles;
  for (int S = kQ8MaxStages; S >= 4; --S) {
    // a warp runs at most S - 1 stages ahead of the slowest one
    int P = (S + per_unit - 1) / per_unit + 2;
    if (P > kQ8MaxSlots) P = kQ8MaxSlots;
    const size_t need = xs + (size_t)P * q8_slot_bytes() + (size_t)S * kStageBytes;
    if (need <= budget && P * per_unit >= S + per_unit) {
      *stages = S;
      *slots = P;
      *smem = need;
      return true;
    }
  }
  return false;
}

cudaError_t launch_q8_project(const void* tiles, int rows, int K, const uint16_t* x, int R,
                              uint16_t* y, uint32_t* status, cudaStream_t s) {
  int S = 0, P = 0;
  size_t smem = 0;
  if (!q8_plan(R, K, &S, &P, &smem)) return cudaErrorInvalidValue;
  Q8Args a{static_cast<const uint8_t*>(tiles), rows, K, R, x, y, status, S, P};
  cudaError_t err = cudaFuncSetAttribute(k_q8_proj, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  int grid = device_sm_count();
  if (grid > rows / 16) grid = rows / 16;
  // a programmatic dependent of the grid before it: the weight stream starts early
  return launch_pdl(k_q8_proj, dim3(grid), kThreads, smem, s, a);
}

}  // namespace dsmoe
