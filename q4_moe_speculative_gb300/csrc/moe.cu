// moe.cu — the speculative-verify Q4 MoE layer: router (K1), gate+up+SwiGLU (K3) and
// down projection with the rank-ordered combine (K4).
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)".
//   paragraph "Decode": the 384-expert router is one dispatch; the shared expert's
//     gate+up+SwiGLU is one kernel; BF16 rounding happens inside the producing kernels.
//   paragraph "DSpark": the decode step is a 6-row verify and the rows share one weight
//     stream.
// Every Q4 weight byte of the shared expert and of the union of routed experts is loaded
// once per call (streaming loads, no reuse across CTAs needed) and applied to every row
// that uses it. All reductions run in a fixed order that does not depend on R or on the
// other rows, so an R-row call writes the same bytes as R one-row calls.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace dsmoe {
namespace {

constexpr int kRouterWarps = 4;
constexpr int kGateUpThreads = 256;
constexpr int kDownThreads = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------------------------
// Activation staging for the Q4 dot products.
//
// A Q4 block is 32 values in 16 bytes: byte j holds value 2j (low nibble) and 2j+1
// (high nibble). The kernels widen a 32-bit word w (values 8m..8m+7) with
//   lo = w & 0x0F0F0F0F  -> values 8m+0, 8m+2, 8m+4, 8m+6
//   hi = (w >> 4) & 0x0F0F0F0F -> values 8m+1, 8m+3, 8m+5, 8m+7
// and one byte-permute per value that builds the fp32 number 128 + nibble exactly
// (exponent byte 0x43, nibble in the top mantissa byte). The activations are therefore
// staged in shared memory in the same order: "chunk" 2m holds the even values of word m
// and chunk 2m+1 the odd ones, 4 floats per chunk, 8 chunks per block. Chunk c of block
// b is stored at chunk position c ^ (b & 7), so that 8 lanes reading 8 consecutive
// blocks with 128-bit loads touch 8 different bank groups.
//
// Because the weights enter as 128 + nibble = q + 136, each block's dot product is
// corrected by 136 * (sum of the block's activations), staged next to the activations.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ int stage_pos(int k) {
  const int blk = k >> 5, w = k & 31;
  const int m = w >> 3, j = (w >> 1) & 3, p = w & 1;
  const int c = 2 * m + p;
  return (blk << 5) + ((c ^ (blk & 7)) << 2) + j;
}

// Stages bf16 row `src` (K values) as fp32 into dst (K floats) and 136 * block sums into
// csum (K / 32 floats). Called by all threads of the CTA; caller synchronises.
__device__ __forceinline__ void stage_row(const uint16_t* __restrict__ src, int K, float* dst,
                                          float* csum, int tid, int nthreads) {
  const uint32_t* s2 = reinterpret_cast<const uint32_t*>(src);
  for (int i = tid; i < K / 2; i += nthreads) {
    const uint32_t w = s2[i];
    dst[stage_pos(2 * i)] = bf16_lo(w);
    dst[stage_pos(2 * i + 1)] = bf16_hi(w);
  }
  for (int blk = tid; blk < K / 32; blk += nthreads) {
    const uint4* p = reinterpret_cast<const uint4*>(src + blk * 32);
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 v = p[c];
      s = __fadd_rn(s, bf16_lo(v.x)); s = __fadd_rn(s, bf16_hi(v.x));
      s = __fadd_rn(s, bf16_lo(v.y)); s = __fadd_rn(s, bf16_hi(v.y));
      s = __fadd_rn(s, bf16_lo(v.z)); s = __fadd_rn(s, bf16_hi(v.z));
      s = __fadd_rn(s, bf16_lo(v.w)); s = __fadd_rn(s, bf16_hi(v.w));
    }
    csum[blk] = __fmul_rn(136.0f, s);
  }
}

// 8 nibbles of w -> 8 floats (128 + nibble), in staged chunk order (even values, odd).
__device__ __forceinline__ void widen8(uint32_t w, float f[8]) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t magic = 0x43000000u;
  f[0] = __uint_as_float(__byte_perm(lo, magic, 0x7044));
  f[1] = __uint_as_float(__byte_perm(lo, magic, 0x7144));
  f[2] = __uint_as_float(__byte_perm(lo, magic, 0x7244));
  f[3] = __uint_as_float(__byte_perm(lo, magic, 0x7344));
  f[4] = __uint_as_float(__byte_perm(hi, magic, 0x7044));
  f[5] = __uint_as_float(__byte_perm(hi, magic, 0x7144));
  f[6] = __uint_as_float(__byte_perm(hi, magic, 0x7244));
  f[7] = __uint_as_float(__byte_perm(hi, magic, 0x7344));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// acc += dot(f[0..7], staged chunks 2m, 2m+1 of block at xb with swizzle sw)
__device__ __forceinline__ float dot8(const float f[8], const float* xb, int m, int sw,
                                      float acc) {
  const float4 a = *reinterpret_cast<const float4*>(xb + (((2 * m) ^ sw) << 2));
  const float4 b = *reinterpret_cast<const float4*>(xb + (((2 * m + 1) ^ sw) << 2));
  acc = __fmaf_rn(f[0], a.x, acc);
  acc = __fmaf_rn(f[1], a.y, acc);
  acc = __fmaf_rn(f[2], a.z, acc);
  acc = __fmaf_rn(f[3], a.w, acc);
  acc = __fmaf_rn(f[4], b.x, acc);
  acc = __fmaf_rn(f[5], b.y, acc);
  acc = __fmaf_rn(f[6], b.z, acc);
  acc = __fmaf_rn(f[7], b.w, acc);
  return acc;
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
  extern __shared__ float smem[];  // x as fp32 [R][H]; then sigmoid scores [R][E]
  __shared__ int s_is_last;
  __shared__ int32_t sel_e[kMaxRows][kMaxTopK];
  __shared__ float sel_s[kMaxRows][kMaxTopK];
  __shared__ uint32_t ubits[kMaxExperts / 32];
  __shared__ int16_t upos[kMaxExperts];
  __shared__ uint32_t u_rowmask[kMaxUnion];
  __shared__ int8_t u_slot[kMaxUnion][8];
  __shared__ int s_nunion;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {
    const uint32_t* x2 = reinterpret_cast<const uint32_t*>(x);
    for (int i = tid; i < R * H / 2; i += blockDim.x) {
      const uint32_t w = x2[i];
      smem[2 * i] = bf16_lo(w);
      smem[2 * i + 1] = bf16_hi(w);
    }
  }
  __syncthreads();

  const int e = blockIdx.x * kRouterWarps + warp;
  if (e < E) {
    float acc[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.0f;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 wv = __ldcs(wrow + c);
      const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                           bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < R) {
          const float4 a = *reinterpret_cast<const float4*>(smem + r * H + c * 8);
          const float4 b = *reinterpret_cast<const float4*>(smem + r * H + c * 8 + 4);
          float t = acc[r];
          t = __fmaf_rn(wf[0], a.x, t); t = __fmaf_rn(wf[1], a.y, t);
          t = __fmaf_rn(wf[2], a.z, t); t = __fmaf_rn(wf[3], a.w, t);
          t = __fmaf_rn(wf[4], b.x, t); t = __fmaf_rn(wf[5], b.y, t);
          t = __fmaf_rn(wf[6], b.z, t); t = __fmaf_rn(wf[7], b.w, t);
          acc[r] = t;
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

  float* s_sm = smem;  // [R][E] sigmoid scores
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
// K3: gate + up + SwiGLU for the shared expert (all rows) and every routed expert of the
// union (its rows). Work unit = (expert slot u, 8 consecutive output rows i), one warp
// per row; lane l reads blocks l, l+32, l+64, l+96 of the gate row and of the up row
// (128-bit streaming loads, each byte once) and applies them to each of the expert's
// rows. h = bf16_rne(silu(g) * u) is written by the producing warp.
// ---------------------------------------------------------------------------------
struct GateUpArgs {
  const uint16_t* x;
  int R, H, I, k;
  Q4Ptr gate, up, sh_gate, sh_up;
  const RouteInfo* route;
  uint16_t* h;
};

__global__ void __launch_bounds__(kGateUpThreads, 2) k3_gate_up(GateUpArgs a) {
  extern __shared__ float smem[];
  const int R = a.R, H = a.H, I = a.I;
  const int nb = H >> 5;
  float* xs = smem;            // [R][H] staged activations
  float* cs = smem + R * H;    // [R][nb] 136 * block sums
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int r = 0; r < R; ++r)
    stage_row(a.x + (size_t)r * H, H, xs + r * H, cs + r * nb, tid, blockDim.x);
  __syncthreads();

  const int n_union = a.route->n_union;
  const int tiles = (I + 7) / 8;
  const int n_units = (1 + n_union) * tiles;
  const size_t row_qs = (size_t)H / 2, row_sc = (size_t)H / 32;

  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const int u = unit / tiles;
    const int i = (unit - u * tiles) * 8 + warp;
    if (i >= I) continue;
    uint32_t rowmask;
    const uint8_t *gq, *uq;
    const uint16_t *gs, *us;
    if (u == 0) {
      rowmask = (1u << R) - 1u;
      gq = a.sh_gate.qs + (size_t)i * row_qs;
      uq = a.sh_up.qs + (size_t)i * row_qs;
      gs = a.sh_gate.sc + (size_t)i * row_sc;
      us = a.sh_up.sc + (size_t)i * row_sc;
    } else {
      const size_t e = (size_t)a.route->expert[u - 1];
      rowmask = a.route->rowmask[u - 1];
      const size_t row = e * I + i;
      gq = a.gate.qs + row * row_qs;
      uq = a.up.qs + row * row_qs;
      gs = a.gate.sc + row * row_sc;
      us = a.up.sc + row * row_sc;
    }

    float ga[kMaxRows], ua[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) { ga[r] = 0.0f; ua[r] = 0.0f; }

    for (int cb = 0; cb < nb; cb += 128) {
      uint4 qg[4], qu[4];
      float sg[4], su[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int blk = cb + 32 * t + lane;
        if (blk < nb) {
          qg[t] = ldg_stream(gq + (size_t)blk * 16);
          qu[t] = ldg_stream(uq + (size_t)blk * 16);
          sg[t] = f16_bits_to_f32(__ldcs(gs + blk));
          su[t] = f16_bits_to_f32(__ldcs(us + blk));
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int blk = cb + 32 * t + lane;
        if (blk < nb) {
          const int sw = blk & 7;
          float bg[kMaxRows], bu[kMaxRows];
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) { bg[r] = 0.0f; bu[r] = 0.0f; }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float fg[8], fu[8];
            widen8(word_of(qg[t], m), fg);
            widen8(word_of(qu[t], m), fu);
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
              if (rowmask & (1u << r)) {
                const float* xb = xs + r * H + blk * 32;
                bg[r] = dot8(fg, xb, m, sw, bg[r]);
                bu[r] = dot8(fu, xb, m, sw, bu[r]);
              }
            }
          }
#pragma unroll
          for (int r = 0; r < kMaxRows; ++r) {
            if (rowmask & (1u << r)) {
              const float c = cs[r * nb + blk];
              ga[r] = __fmaf_rn(sg[t], __fsub_rn(bg[r], c), ga[r]);
              ua[r] = __fmaf_rn(su[t], __fsub_rn(bu[r], c), ua[r]);
            }
          }
        }
      }
    }

#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (rowmask & (1u << r)) {
        const float g = warp_sum(ga[r]);
        const float uu = warp_sum(ua[r]);
        if (lane == r) {
          const int slot = (u == 0) ? 0 : a.route->slot[u - 1][r];
          const float silu = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
          a.h[((size_t)r * (1 + a.k) + slot) * I + i] = f32_to_bf16_rne(__fmul_rn(silu, uu));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------
// K4: down projection + combine. Work unit = (expert slot u, tile of 64 output rows of
// H). The CTA stages h of the expert's rows (fp32, same layout as K3's activations);
// each warp computes 8 output rows, 4 at a time with 8 lanes per row (lane j of a group
// reads blocks j, j+8, j+16, j+24 of its row), and writes fp32 partials per (row, slot).
// The last unit to finish a tile (arrival count, no waiting) forms
//   y = bf16_rne(o_shared + sum_j w_j o_j)   in rank order j.
// ---------------------------------------------------------------------------------
struct DownArgs {
  const uint16_t* h;
  int R, H, I, k;
  Q4Ptr down, sh_down;
  const RouteInfo* route;
  const float* topk_w;
  float* opart;
  uint32_t* tile_count;
  uint16_t* y;
};

__global__ void __launch_bounds__(kDownThreads) k4_down(DownArgs a) {
  extern __shared__ float smem[];
  __shared__ int s_last;
  const int R = a.R, H = a.H, I = a.I, k = a.k;
  const int nb = I >> 5;
  float* hs = smem;            // [R][I]
  float* cs = smem + R * I;    // [R][nb]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 3, gl = lane & 7;

  const int n_exp = 1 + a.route->n_union;
  const int tiles = (H + kDownTileH - 1) / kDownTileH;
  const int n_units = n_exp * tiles;
  const int beg = (int)(((long long)blockIdx.x * n_units) / gridDim.x);
  const int end = (int)(((long long)(blockIdx.x + 1) * n_units) / gridDim.x);
  const size_t row_qs = (size_t)I / 2, row_sc = (size_t)I / 32;

  int staged = -1;
  uint32_t rowmask = 0;
  int slot[kMaxRows];
  for (int unit = beg; unit < end; ++unit) {
    const int u = unit / tiles;
    const int tile = unit - u * tiles;
    if (u != staged) {
      __syncthreads();
      if (u == 0) {
        rowmask = (1u << R) - 1u;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) slot[r] = 0;
      } else {
        rowmask = a.route->rowmask[u - 1];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) slot[r] = a.route->slot[u - 1][r];
      }
      for (int r = 0; r < R; ++r)
        if (rowmask & (1u << r))
          stage_row(a.h + ((size_t)r * (1 + k) + slot[r]) * I, I, hs + r * I, cs + r * nb,
                    tid, blockDim.x);
      __syncthreads();
      staged = u;
    }
    const uint8_t* dq;
    const uint16_t* dsc;
    if (u == 0) {
      dq = a.sh_down.qs;
      dsc = a.sh_down.sc;
    } else {
      const size_t e = (size_t)a.route->expert[u - 1];
      dq = a.down.qs + e * H * row_qs;
      dsc = a.down.sc + e * H * row_sc;
    }
    const int hr0 = tile * kDownTileH + warp * 8;

    float acc[2][kMaxRows];
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) acc[s][r] = 0.0f;

    for (int cb = 0; cb < nb; cb += 32) {
      uint4 q[2][4];
      float sc[2][4];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int hr = hr0 + 4 * s + grp;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int blk = cb + gl + 8 * t;
          if (hr < H && blk < nb) {
            q[s][t] = ldg_stream(dq + (size_t)hr * row_qs + (size_t)blk * 16);
            sc[s][t] = f16_bits_to_f32(__ldcs(dsc + (size_t)hr * row_sc + blk));
          }
        }
      }
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int hr = hr0 + 4 * s + grp;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int blk = cb + gl + 8 * t;
          if (hr < H && blk < nb) {
            const int sw = blk & 7;
            float b[kMaxRows];
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) b[r] = 0.0f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              float f[8];
              widen8(word_of(q[s][t], m), f);
#pragma unroll
              for (int r = 0; r < kMaxRows; ++r)
                if (rowmask & (1u << r)) b[r] = dot8(f, hs + r * I + blk * 32, m, sw, b[r]);
            }
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r)
              if (rowmask & (1u << r))
                acc[s][r] = __fmaf_rn(sc[s][t], __fsub_rn(b[r], cs[r * nb + blk]), acc[s][r]);
          }
        }
      }
    }

#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int hr = hr0 + 4 * s + grp;
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (rowmask & (1u << r)) {
          float v = acc[s][r];
          v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
          if (gl == 0 && hr < H) a.opart[((size_t)r * (1 + k) + slot[r]) * H + hr] = v;
        }
      }
    }

    // Tile arrival; the last expert unit of this tile combines it.
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned prev = atomicAdd(&a.tile_count[tile], 1u);
      s_last = (prev == (unsigned)(n_exp - 1));
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int idx = tid; idx < R * kDownTileH; idx += blockDim.x) {
        const int r = idx / kDownTileH;
        const int hr = tile * kDownTileH + (idx - r * kDownTileH);
        if (hr >= H) continue;
        const float* orow = a.opart + (size_t)r * (1 + k) * H + hr;
        float y = __ldcg(orow);
        for (int j = 0; j < k; ++j)
          y = __fmaf_rn(a.topk_w[r * k + j], __ldcg(orow + (size_t)(1 + j) * H), y);
        a.y[(size_t)r * H + hr] = f32_to_bf16_rne(y);
      }
    }
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

MoeLayout moe_layout(const MoeDims& d) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  MoeLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  L.tile_count = off; off += up(sizeof(uint32_t) * (size_t)((d.H + kDownTileH - 1) / kDownTileH));
  L.zero_bytes = off;
  L.logits = off; off += up(sizeof(float) * (size_t)d.R * d.E);
  L.route = off; off += up(sizeof(RouteInfo));
  L.h = off; off += up(sizeof(uint16_t) * (size_t)d.R * (1 + d.k) * d.I);
  L.opart = off; off += up(sizeof(float) * (size_t)d.R * (1 + d.k) * d.H);
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
  const size_t smem = sizeof(float) * ((size_t)d.R * d.H + (size_t)d.R * (d.H / 32));
  cudaError_t err = set_smem(k3_gate_up, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k3_gate_up, kGateUpThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int tiles = (d.I + 7) / 8;
  const int max_units = (1 + d.R * d.k) * tiles;
  int grid = device_sm_count() * per_sm;
  if (grid > max_units) grid = max_units;
  GateUpArgs a{x, d.R, d.H, d.I, d.k, gate, up, sh_gate, sh_up, ws.route, ws.h};
  k3_gate_up<<<grid, kGateUpThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_down(const MoeDims& d, Q4Ptr down, Q4Ptr sh_down, const float* topk_w,
                        uint16_t* y, const MoeWorkspace& ws, cudaStream_t s) {
  const size_t smem = sizeof(float) * ((size_t)d.R * d.I + (size_t)d.R * (d.I / 32));
  cudaError_t err = set_smem(k4_down, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k4_down, kDownThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int tiles = (d.H + kDownTileH - 1) / kDownTileH;
  const int min_units = tiles;  // at least the shared expert
  int grid = device_sm_count() * per_sm;
  if (grid > min_units * 4) grid = min_units * 4 > 0 ? min_units * 4 : 1;
  DownArgs a{ws.h, d.R, d.H, d.I, d.k, down, sh_down, ws.route, topk_w, ws.opart,
             ws.tile_count, y};
  k4_down<<<grid, kDownThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsmoe
