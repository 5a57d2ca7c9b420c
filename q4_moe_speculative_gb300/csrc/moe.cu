// moe.cu — the speculative-verify Q4 MoE layer: router (K1), gate+up+SwiGLU (K3) and
// down projection with the rank-ordered combine (K4).
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
// Weight tiles stream through a per-warp cp.async ring in shared memory (4 stages), so no
// register holds data in flight; units of work are taken from a counter (work stealing).
#include <climits>
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace dsmoe {
namespace {

constexpr int kRouterWarps = 8;
constexpr int kMmaWarps = 16;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kStages = 4;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- PTX helpers --------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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
// K1: router. One warp per expert computes z = x . Wr[e] for all R rows (fp32, lane-
// strided partial sums then a butterfly), the last CTA to finish (atomic arrival count,
// no waiting) computes sigmoid scores, the top-k per row, the renormalised weights and
// the union of the selected experts with each one's rows and rank slots.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouterWarps * 32)
    k1_router(const uint16_t* __restrict__ x, int R, int H, const uint16_t* __restrict__ wr,
              int E, int k, float* __restrict__ logits, int32_t* __restrict__ topk_idx,
              float* __restrict__ topk_w, RouteInfo* __restrict__ route, WsHeader* hdr) {
  extern __shared__ float smem_f[];  // x as fp32 [R][H]; then sigmoid scores [R][E]
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
  {
    // 8 values per 16-byte load; loads of an unrolled batch are independent, so the CTA
    // has many in flight instead of one load -> store round trip at a time.
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    const int n8 = R * H / 8;
#pragma unroll 8
    for (int i = tid; i < n8; i += blockDim.x) {
      const uint4 v = __ldg(x8 + i);
      float4* d = reinterpret_cast<float4*>(smem_f + 8 * i);
      d[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
      d[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
    }
  }
  __syncthreads();

  const int e = blockIdx.x * kRouterWarps + warp;
  if (e < E) {
    float acc[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.0f;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    const int nc = H / 8;
    // All of a warp's weight loads for up to 4096 values are issued before any use.
    for (int c0 = 0; c0 < nc; c0 += 16 * 32) {
      uint4 wv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = c0 + u * 32 + lane;
        wv[u] = c < nc ? __ldcs(wrow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c >= nc) continue;
        const float wf[8] = {bf16_lo(wv[u].x), bf16_hi(wv[u].x), bf16_lo(wv[u].y),
                             bf16_hi(wv[u].y), bf16_lo(wv[u].z), bf16_hi(wv[u].z),
                             bf16_lo(wv[u].w), bf16_hi(wv[u].w)};
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
          if (r < R) {
            const float4 a = *reinterpret_cast<const float4*>(smem_f + r * H + c * 8);
            const float4 b = *reinterpret_cast<const float4*>(smem_f + r * H + c * 8 + 4);
            float t = acc[r];
            t = __fmaf_rn(wf[0], a.x, t); t = __fmaf_rn(wf[1], a.y, t);
            t = __fmaf_rn(wf[2], a.z, t); t = __fmaf_rn(wf[3], a.w, t);
            t = __fmaf_rn(wf[4], b.x, t); t = __fmaf_rn(wf[5], b.y, t);
            t = __fmaf_rn(wf[6], b.z, t); t = __fmaf_rn(wf[7], b.w, t);
            acc[r] = t;
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < R) {
        const float z = warp_sum(acc[r]);
        if (lane == 0) logits[r * E + e] = z;
      }
    }
  }

  // Arrival count: the last CTA continues, the others are done. Nobody waits.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&hdr->router_arrivals, 1u);
    s_is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_is_last) return;
  __threadfence();

  float* s_sm = smem_f;  // [R][E] sigmoid scores
  for (int i = tid; i < R * E; i += blockDim.x) {
    const float z = __ldcg(logits + i);
    s_sm[i] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-z)));
  }
  if (tid < kMaxExperts / 32) ubits[tid] = 0u;
  __syncthreads();

  for (int r = warp; r < R; r += kRouterWarps) {
    float* sr = s_sm + r * E;
    for (int j = 0; j < k; ++j) {
      float best = -1.0f;
      int bi = INT_MAX;
      for (int e2 = lane; e2 < E; e2 += 32) {
        const float v = sr[e2];
        if (v > best) { best = v; bi = e2; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
      }
      if (lane == 0) {
        sel_e[r][j] = bi;
        sel_s[r][j] = best;
        sr[bi] = -1.0f;  // taken (scores are >= 0)
      }
      __syncwarp();
    }
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
// K3: gate + up + SwiGLU. Unit of work = (expert slot u, 16 rows of I, one of KP parts of
// K); expert slot 0 is the shared expert (all rows), slot u >= 1 the u-th expert of the
// union (its rows). A warp streams its unit's gate and up rows in tiles of 4 Q4 blocks
// through its cp.async ring and accumulates D[16 rows][8 cols] with mma.sync; the
// activations sit in shared memory as bf16 in MMA pair order (staged once per CTA).
// The last of the KP parts to arrive (atomic count) adds the parts in a fixed order and
// writes h = bf16_rne(silu(g) * u) for the expert's rows.
// ---------------------------------------------------------------------------------
struct GuStage {
  uint32_t a[2][4][16][4];   // [gate/up][block j][row][word]
  uint32_t s[2][16][2];      // [gate/up][row][4 fp16 scales]
};

struct GateUpArgs {
  const uint16_t* x;
  int R, H, I, k;
  Q4Ptr gate, up, sh_gate, sh_up;
  const RouteInfo* route;
  uint16_t* h;
  float* part;               // [(1+R*k) * (I/16) * KP][32 lanes][8]
  uint32_t* part_count;      // [(1+R*k) * (I/16)]
  uint32_t* unit_counter;
};


__global__ void __launch_bounds__(kMmaThreads, 1) k3_gate_up(GateUpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int R = a.R, H = a.H, I = a.I, k = a.k;
  const int nb = H >> 5;                        // Q4 blocks per row
  const int T = (nb + 3) >> 2;                  // tiles of 4 blocks
  const int TP = (T + 3) >> 2;                  // tiles per K part
  const int KP = (T + TP - 1) / TP;             // K parts (<= 4)
  const int RT = I >> 4;                        // 16-row tiles
  const int xstride = H * 2 + 64;               // bytes per staged activation row
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;

  uint8_t* xs = smem;
  GuStage* stages = reinterpret_cast<GuStage*>(smem + ((R * xstride + 127) & ~127)) + warp * kStages;
  int* wdesc = reinterpret_cast<int*>(reinterpret_cast<GuStage*>(smem + ((R * xstride + 127) & ~127)) +
                                      kMmaWarps * kStages) + warp * (2 * kStages);

  // Activations -> shared memory, bf16 in MMA pair order (independent of the router).
#pragma unroll 4
  for (int i = tid; i < R * (H >> 3); i += blockDim.x) {
    const int r = i / (H >> 3), grp = i - r * (H >> 3);
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + (size_t)r * H + grp * 8);
    *reinterpret_cast<uint4*>(xs + r * xstride + (grp >> 2) * 64 + (grp & 3) * 16) = pair_order(v);
  }
  __syncthreads();
  pdl_wait();   // the route produced by the router grid is visible from here on

  const RouteInfo* rt_info = a.route;
  const int n_union = rt_info->n_union;
  const int n_units = (1 + n_union) * RT * KP;
  const size_t row_qs = (size_t)H / 2, row_sc = (size_t)nb;

  // Issue cursor (warp-uniform). A unit is decoded once, when the warp takes it; each
  // further tile only advances the source pointers.
  int iu = -1, it = 0, itiles = 0, iblk = 0;
  bool exhausted = false;
  const uint8_t *igq = nullptr, *iuq = nullptr;
  const uint16_t *igs = nullptr, *ius = nullptr;

  auto issue = [&](int stage) {
    int unit = -1, tile = 0;
    if (!exhausted && (iu < 0 || it >= itiles)) {
      int nu = 0;
      if (lane == 0) nu = (int)atomicAdd(a.unit_counter, 1u);
      nu = __shfl_sync(0xffffffffu, nu, 0);
      if (nu >= n_units) {
        exhausted = true;
      } else {
        iu = nu;
        it = 0;
        const int u = nu / (RT * KP);
        const int rem = nu - u * RT * KP;
        const int rti = rem / KP, kp = rem - rti * KP;
        itiles = min(TP, T - kp * TP);
        iblk = kp * TP * 4;
        const size_t row0 = (size_t)rti * 16;
        if (u == 0) {
          igq = a.sh_gate.qs + row0 * row_qs; iuq = a.sh_up.qs + row0 * row_qs;
          igs = a.sh_gate.sc + row0 * row_sc; ius = a.sh_up.sc + row0 * row_sc;
        } else {
          const size_t e = (size_t)rt_info->expert[u - 1];
          igq = a.gate.qs + (e * I + row0) * row_qs; iuq = a.up.qs + (e * I + row0) * row_qs;
          igs = a.gate.sc + (e * I + row0) * row_sc; ius = a.up.sc + (e * I + row0) * row_sc;
        }
      }
    }
    if (!exhausted) {
      unit = iu;
      tile = it++;
    }
    if (lane == 0) {
      wdesc[2 * stage] = unit;
      wdesc[2 * stage + 1] = tile;
    }
    if (unit >= 0) {
      const int blk0 = iblk + tile * 4;
      GuStage& S = stages[stage];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int pp = lane + 32 * h2;
        const int row = pp & 15, j = pp >> 4;
        const bool v = blk0 + j < nb;
        const size_t off = row * row_qs + (size_t)(blk0 + j) * 16;
        cp_async16(&S.a[0][j][row][0], v ? igq + off : igq, v);
        cp_async16(&S.a[1][j][row][0], v ? iuq + off : iuq, v);
      }
      {
        const int row = lane >> 1, hf = lane & 1;
        const bool v = blk0 + 2 * hf < nb;
        const size_t off = row * row_sc + blk0 + 2 * hf;
        cp_async4(&S.s[0][row][hf], v ? igs + off : igs, v);
        cp_async4(&S.s[1][row][hf], v ? ius + off : ius, v);
      }
    }
    cp_async_commit();
  };

  float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue(s);

  // Compute cursor: the unit of the tile being computed, decoded once per unit.
  int cu = -1, u = 0, rti = 0, kp = 0, tiles = 0;
  uint32_t rowmask = 0;
  bool member = false;
  for (int t = 0;; ++t) {
    issue((t + kStages - 1) % kStages);
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const int stage = t % kStages;
    const int unit = wdesc[2 * stage], tile = wdesc[2 * stage + 1];
    if (unit < 0) break;
    if (unit != cu) {
      cu = unit;
      u = unit / (RT * KP);
      const int rem = unit - u * RT * KP;
      rti = rem / KP;
      kp = rem - rti * KP;
      tiles = min(TP, T - kp * TP);
      rowmask = (u == 0) ? ((1u << R) - 1u) : rt_info->rowmask[u - 1];
      member = (g < R) && ((rowmask >> g) & 1u);
    }
    if (tile == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) { ag[i] = 0.f; au[i] = 0.f; }
    }
    const GuStage& S = stages[stage];
    const int blk0 = (kp * TP + tile) * 4;
    // fp16 scales of this lane's rows g and g+8 for the tile's 4 blocks, widened once
    const uint2 sgv0 = *reinterpret_cast<const uint2*>(&S.s[0][g][0]);
    const uint2 sgv8 = *reinterpret_cast<const uint2*>(&S.s[0][g + 8][0]);
    const uint2 suv0 = *reinterpret_cast<const uint2*>(&S.s[1][g][0]);
    const uint2 suv8 = *reinterpret_cast<const uint2*>(&S.s[1][g + 8][0]);
    float sg0[4], sg8[4], su0[4], su8[4];
    widen_scales(sgv0, sg0); widen_scales(sgv8, sg8);
    widen_scales(suv0, su0); widen_scales(suv8, su8);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int blk = blk0 + j;
      if (blk < nb) {
        const uint4 X = member ? *reinterpret_cast<const uint4*>(xs + g * xstride + blk * 64 + q * 16)
                               : make_uint4(0, 0, 0, 0);
        float d[4];
        q4_block_mma(S.a[0][j][g][q], S.a[0][j][g + 8][q], X, d);
        ag[0] = __fmaf_rn(sg0[j], d[0], ag[0]); ag[1] = __fmaf_rn(sg0[j], d[1], ag[1]);
        ag[2] = __fmaf_rn(sg8[j], d[2], ag[2]); ag[3] = __fmaf_rn(sg8[j], d[3], ag[3]);
        q4_block_mma(S.a[1][j][g][q], S.a[1][j][g + 8][q], X, d);
        au[0] = __fmaf_rn(su0[j], d[0], au[0]); au[1] = __fmaf_rn(su0[j], d[1], au[1]);
        au[2] = __fmaf_rn(su8[j], d[2], au[2]); au[3] = __fmaf_rn(su8[j], d[3], au[3]);
      }
    }
    __syncwarp();

    if (tile == tiles - 1) {
      // All K parts of (u, row tile) in a fixed order, then the SwiGLU epilogue.
      float sg[4], su[4];
      bool last = true;
      const int ut = u * RT + rti;
      if (KP > 1) {
        float* mine = a.part + ((size_t)ut * KP + kp) * 256 + lane * 8;
        *reinterpret_cast<float4*>(mine) = make_float4(ag[0], ag[1], ag[2], ag[3]);
        *reinterpret_cast<float4*>(mine + 4) = make_float4(au[0], au[1], au[2], au[3]);
        __threadfence();
        __syncwarp();
        unsigned prev = 0;
        if (lane == 0) prev = atomicAdd(a.part_count + ut, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        last = (prev == (unsigned)(KP - 1));
        if (last) {
          __threadfence();
#pragma unroll
          for (int i = 0; i < 4; ++i) { sg[i] = 0.f; su[i] = 0.f; }
          for (int p = 0; p < KP; ++p) {
            const float* src = a.part + ((size_t)ut * KP + p) * 256 + lane * 8;
            const float4 g4 = __ldcg(reinterpret_cast<const float4*>(src));
            const float4 u4 = __ldcg(reinterpret_cast<const float4*>(src + 4));
            sg[0] = __fadd_rn(sg[0], g4.x); sg[1] = __fadd_rn(sg[1], g4.y);
            sg[2] = __fadd_rn(sg[2], g4.z); sg[3] = __fadd_rn(sg[3], g4.w);
            su[0] = __fadd_rn(su[0], u4.x); su[1] = __fadd_rn(su[1], u4.y);
            su[2] = __fadd_rn(su[2], u4.z); su[3] = __fadd_rn(su[3], u4.w);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) { sg[i] = ag[i]; su[i] = au[i]; }
      }
      if (last) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 2 * q + (e & 1);
          const int row = rti * 16 + g + ((e & 2) ? 8 : 0);
          if (c < R && ((rowmask >> c) & 1u)) {
            const int slot = (u == 0) ? 0 : rt_info->slot[u - 1][c];
            const float gv = sg[e];
            const float silu = __fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv)));
            a.h[((size_t)c * (1 + k) + slot) * I + row] = f32_to_bf16_rne(__fmul_rn(silu, su[e]));
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  pdl_trigger();
}

// ---------------------------------------------------------------------------------
// K4: down projection + combine. Unit of work = (expert slot u, 32 rows of H), all of K
// = I. The warp streams the down rows and the expert's h (its rows' slots) through a
// 3-stage cp.async ring; each staged h fragment feeds the MMAs of both 16-row halves.
// It writes fp32 partials per (row, slot); the last unit to finish a 32-row tile
// (arrival count, no waiting) forms  y = bf16_rne(o_shared + sum_j w_j o_j)  in rank
// order j.
// ---------------------------------------------------------------------------------
constexpr int kDownStages = 3;
constexpr int kDownRows = 32;

struct DnStage {
  uint32_t a[4][kDownRows][4];   // [block j][row][word]
  uint32_t s[kDownRows][2];      // [row][4 fp16 scales]
  uint4 b[4][32];                // [block j][lane]: h values 8q..8q+7 of verify row g
};

struct DownArgs {
  const uint16_t* h;
  int R, H, I, k;
  Q4Ptr down, sh_down;
  const RouteInfo* route;
  const float* topk_w;
  float* opart;
  uint32_t* tile_count;      // [H/32]
  uint32_t* unit_counter;
  uint16_t* y;
};

__global__ void __launch_bounds__(kMmaThreads, 1) k4_down(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int R = a.R, H = a.H, I = a.I, k = a.k;
  const int nb = I >> 5;
  const int T = (nb + 3) >> 2;
  const int RT = H / kDownRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  DnStage* stages = reinterpret_cast<DnStage*>(smem) + warp * kDownStages;
  int* wdesc = reinterpret_cast<int*>(reinterpret_cast<DnStage*>(smem) + kMmaWarps * kDownStages) +
               warp * (2 * kDownStages);

  pdl_wait();   // h and the route are complete from here on
  const RouteInfo* rt_info = a.route;
  const int n_exp = 1 + rt_info->n_union;
  const int n_units = n_exp * RT;
  const size_t row_qs = (size_t)I / 2, row_sc = (size_t)nb;

  int iu = -1, it = 0;
  bool exhausted = false;
  const uint8_t* idq = nullptr;
  const uint16_t* ids = nullptr;
  const uint16_t* ihrow = nullptr;
  bool imember = false;
  auto issue = [&](int stage) {
    int unit = -1, tile = 0;
    if (!exhausted && (iu < 0 || it >= T)) {
      int nu = 0;
      if (lane == 0) nu = (int)atomicAdd(a.unit_counter, 1u);
      nu = __shfl_sync(0xffffffffu, nu, 0);
      if (nu >= n_units) {
        exhausted = true;
      } else {
        iu = nu;
        it = 0;
        const int u = nu / RT, rti = nu - u * RT;
        const size_t row0 = (size_t)rti * kDownRows;
        uint32_t rowmask;
        int slot_g = 0;
        if (u == 0) {
          idq = a.sh_down.qs + row0 * row_qs;
          ids = a.sh_down.sc + row0 * row_sc;
          rowmask = (1u << R) - 1u;
        } else {
          const size_t e = (size_t)rt_info->expert[u - 1];
          idq = a.down.qs + (e * H + row0) * row_qs;
          ids = a.down.sc + (e * H + row0) * row_sc;
          rowmask = rt_info->rowmask[u - 1];
          slot_g = rt_info->slot[u - 1][g];
        }
        imember = (g < R) && ((rowmask >> g) & 1u);
        ihrow = a.h + ((size_t)g * (1 + k) + (imember ? slot_g : 0)) * I;
      }
    }
    if (!exhausted) {
      unit = iu;
      tile = it++;
    }
    if (lane == 0) {
      wdesc[2 * stage] = unit;
      wdesc[2 * stage + 1] = tile;
    }
    if (unit >= 0) {
      const int blk0 = tile * 4;
      DnStage& S = stages[stage];
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        const int pp = lane + 32 * h4;
        const int row = pp & (kDownRows - 1), j = pp >> 5;
        const bool v = blk0 + j < nb;
        cp_async16(&S.a[j][row][0], v ? idq + row * row_qs + (size_t)(blk0 + j) * 16 : idq, v);
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int pp = lane + 32 * h2;
        const int row = pp >> 1, hf = pp & 1;
        const bool v = blk0 + 2 * hf < nb;
        cp_async4(&S.s[row][hf], v ? ids + row * row_sc + blk0 + 2 * hf : ids, v);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool v = imember && (blk0 + j < nb);
        cp_async16(&S.b[j][lane], v ? ihrow + (blk0 + j) * 32 + q * 8 : a.h, v);
      }
    }
    cp_async_commit();
  };

  float acc[2][4];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[hh][i] = 0.f;
#pragma unroll
  for (int s = 0; s < kDownStages - 1; ++s) issue(s);

  int cu = -1, u = 0, rti = 0;
  for (int t = 0;; ++t) {
    issue((t + kDownStages - 1) % kDownStages);
    cp_async_wait<kDownStages - 1>();
    __syncwarp();
    const int stage = t % kDownStages;
    const int unit = wdesc[2 * stage], tile = wdesc[2 * stage + 1];
    if (unit < 0) break;
    if (unit != cu) {
      cu = unit;
      u = unit / RT;
      rti = unit - u * RT;
    }
    if (tile == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[hh][i] = 0.f;
    }
    const DnStage& S = stages[stage];
    const int blk0 = tile * 4;
    float sf[2][2][4];   // [half][row g / g+8][block]
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      widen_scales(*reinterpret_cast<const uint2*>(&S.s[hh * 16 + g][0]), sf[hh][0]);
      widen_scales(*reinterpret_cast<const uint2*>(&S.s[hh * 16 + g + 8][0]), sf[hh][1]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (blk0 + j < nb) {
        const uint4 X = pair_order(S.b[j][lane]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float d[4];
          q4_block_mma(S.a[j][hh * 16 + g][q], S.a[j][hh * 16 + g + 8][q], X, d);
          acc[hh][0] = __fmaf_rn(sf[hh][0][j], d[0], acc[hh][0]);
          acc[hh][1] = __fmaf_rn(sf[hh][0][j], d[1], acc[hh][1]);
          acc[hh][2] = __fmaf_rn(sf[hh][1][j], d[2], acc[hh][2]);
          acc[hh][3] = __fmaf_rn(sf[hh][1][j], d[3], acc[hh][3]);
        }
      }
    }
    __syncwarp();

    if (tile == T - 1) {
      const uint32_t rowmask = (u == 0) ? ((1u << R) - 1u) : rt_info->rowmask[u - 1];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 2 * q + (e & 1);
          const int row = rti * kDownRows + hh * 16 + g + ((e & 2) ? 8 : 0);
          if (c < R && ((rowmask >> c) & 1u)) {
            const int slot = (u == 0) ? 0 : rt_info->slot[u - 1][c];
            a.opart[((size_t)c * (1 + k) + slot) * H + row] = acc[hh][e];
          }
        }
      }
      __threadfence();
      __syncwarp();
      unsigned prev = 0;
      if (lane == 0) prev = atomicAdd(a.tile_count + rti, 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == (unsigned)(n_exp - 1)) {
        __threadfence();
        for (int idx = lane; idx < R * kDownRows; idx += 32) {
          const int r = idx / kDownRows, row = rti * kDownRows + (idx % kDownRows);
          const float* orow = a.opart + (size_t)r * (1 + k) * H + row;
          float yv = __ldcg(orow);
          for (int j = 0; j < k; ++j)
            yv = __fmaf_rn(a.topk_w[r * k + j], __ldcg(orow + (size_t)(1 + j) * H), yv);
          a.y[(size_t)r * H + row] = f32_to_bf16_rne(yv);
        }
      }
    }
  }
  cp_async_wait<0>();
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename... Exp, typename... Act>
cudaError_t launch_pdl(void (*kernel)(Exp...), int grid, int block, size_t smem, cudaStream_t s,
                       Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

size_t gate_up_smem(const MoeDims& d) {
  const size_t xbytes = ((size_t)d.R * (d.H * 2 + 64) + 127) & ~(size_t)127;
  return xbytes + sizeof(GuStage) * kMmaWarps * kStages + sizeof(int) * 2 * kStages * kMmaWarps;
}

size_t down_smem() {
  return sizeof(DnStage) * kMmaWarps * kDownStages + sizeof(int) * 2 * kDownStages * kMmaWarps;
}

}  // namespace

size_t gate_up_smem_bytes(const MoeDims& d) { return gate_up_smem(d); }

int gate_up_kparts(int H) {
  const int T = ((H >> 5) + 3) >> 2;
  const int TP = (T + 3) >> 2;
  return (T + TP - 1) / TP;
}

MoeLayout moe_layout(const MoeDims& d) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t U = 1 + (size_t)d.R * d.k;           // expert slots (shared + union bound)
  const size_t RT = (size_t)d.I / 16;
  MoeLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  L.tile_count = off; off += up(sizeof(uint32_t) * (size_t)(d.H / 16));
  L.part_count = off; off += up(sizeof(uint32_t) * U * RT);
  L.zero_bytes = off;
  L.logits = off; off += up(sizeof(float) * (size_t)d.R * d.E);
  L.route = off; off += up(sizeof(RouteInfo));
  L.h = off; off += up(sizeof(uint16_t) * (size_t)d.R * (1 + d.k) * d.I);
  L.opart = off; off += up(sizeof(float) * (size_t)d.R * (1 + d.k) * d.H);
  L.part = off; off += up(sizeof(float) * U * RT * (size_t)gate_up_kparts(d.H) * 256);
  L.total = off;
  return L;
}

cudaError_t launch_router(const MoeDims& d, const uint16_t* x, const uint16_t* router_w,
                          int32_t* topk_idx, float* topk_w, const MoeWorkspace& ws,
                          cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)d.R * (size_t)(d.H > d.E ? d.H : d.E);
  cudaError_t err = set_smem(k1_router, smem);
  if (err != cudaSuccess) return err;
  const int grid = (d.E + kRouterWarps - 1) / kRouterWarps;
  k1_router<<<grid, kRouterWarps * 32, smem, s>>>(
      x, d.R, d.H, router_w, d.E, d.k, ws.logits, topk_idx, topk_w, ws.route,
      reinterpret_cast<WsHeader*>(ws.header));
  return cudaGetLastError();
}

cudaError_t launch_gate_up(const MoeDims& d, const uint16_t* x, Q4Ptr gate, Q4Ptr up,
                           Q4Ptr sh_gate, Q4Ptr sh_up, const MoeWorkspace& ws,
                           cudaStream_t s) {
  const size_t smem = gate_up_smem(d);
  cudaError_t err = set_smem(k3_gate_up, smem);
  if (err != cudaSuccess) return err;
  GateUpArgs a{x, d.R, d.H, d.I, d.k, gate, up, sh_gate, sh_up, ws.route, ws.h, ws.part,
               ws.part_count, ws.header + 2};
  return launch_pdl(k3_gate_up, device_sm_count(), kMmaThreads, smem, s, a);
}

cudaError_t launch_down(const MoeDims& d, Q4Ptr down, Q4Ptr sh_down, const float* topk_w,
                        uint16_t* y, const MoeWorkspace& ws, cudaStream_t s) {
  const size_t smem = down_smem();
  cudaError_t err = set_smem(k4_down, smem);
  if (err != cudaSuccess) return err;
  DownArgs a{ws.h, d.R, d.H, d.I, d.k, down, sh_down, ws.route, topk_w, ws.opart,
             ws.tile_count, ws.header + 3, y};
  return launch_pdl(k4_down, device_sm_count(), kMmaThreads, smem, s, a);
}

}  // namespace dsmoe
