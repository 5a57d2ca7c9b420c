// attn.cu — sparse attention over the selected blocks: each verify row's query heads attend
// to the tokens of the blocks the top-k selection picked for that row and layer.
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)", paragraph
// "Decode at depth": compressed attention picks 512 blocks per layer, and attention reads
// only those. The attention arithmetic itself is not on the pages; this is the plain
// reading: for row r and head h, s_t = q_{r,h} . k_t / sqrt(D) over the tokens t of the
// selected blocks (all heads of a row share the token's key and value), p = softmax(s),
// o = sum_t p_t v_t, rounded once to bf16.
//
// k_attn: CTA = (split of the row's selection, layer x row); 4 warps, each taking groups of
// 16 selected tokens (16 / block_tokens selection entries) in turn. A group's keys and
// values (256 bytes each per token) are gathered by cp.async into the warp's double buffer
// (272-byte rows). S = Q K^T and O += P V run as mma.sync m16n8k16 (bf16 in, fp32
// accumulate): the up to 16 heads are the M dimension, Q stays in registers, K^T and V
// fragments come from ldmatrix (V transposed). P is split into a bf16 high and low part so
// that the P V products keep about 16 bits of P. The running max, normaliser and output
// follow the online softmax; the warps' states are merged in warp order, the splits' states
// in split order by the CTA that finishes a row last.
#include "common.cuh"
#include "kernels.h"

namespace dsmoe {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kD = 128;
constexpr int kGroup = 16;                    // tokens per warp step
constexpr int kPitch = 272;                   // bytes per staged token row
constexpr int kBufBytes = 2 * kGroup * kPitch;   // keys + values of one group
constexpr int kSmem = kWarps * 2 * kBufBytes;    // double buffer per warp
constexpr float kNegInf = -INFINITY;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// bf16 pair of (lo, hi) rounded to nearest, and the pair of what rounding left over.
__device__ __forceinline__ void split_pair(float lo, float hi, uint32_t* big, uint32_t* rest) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  const float2 bf = __bfloat1622float2(b);
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo - bf.x, hi - bf.y);
  *big = *reinterpret_cast<const uint32_t*>(&b);
  *rest = *reinterpret_cast<const uint32_t*>(&r);
}

struct AttnArgs {
  int L, R, Hq, N, bs, K;     // layers, rows, heads, blocks, tokens per block, sel width
  int64_t kv_stride;          // values between layers of k / v
  const uint16_t* q;          // [L][R][Hq][128]
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* sel;         // [L][R][K]
  uint16_t* out;              // [L][R][Hq][128]
  float* part;                // [splits][L R][16][130]: max, normaliser, 128 outputs
  int32_t* count;             // [L R] CTAs of the row finished
  uint32_t* status;
  int splits;
};

__global__ void __launch_bounds__(kThreads) k_attn(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ int s_last;
  const int sp = blockIdx.x, lr = blockIdx.y, l = lr / a.R;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int per_group = kGroup / a.bs;            // selection entries per group
  const int groups = (a.K + per_group - 1) / per_group;
  const int gb = (int)(((long long)sp * groups) / a.splits);
  const int ge = (int)(((long long)(sp + 1) * groups) / a.splits);
  const int32_t* sel = a.sel + (size_t)lr * a.K;
  const uint8_t* kl = reinterpret_cast<const uint8_t*>(a.k + (size_t)l * a.kv_stride);
  const uint8_t* vl = reinterpret_cast<const uint8_t*>(a.v + (size_t)l * a.kv_stride);
  const int nblk = a.N;

  // Q fragments (heads g and g + 8 of this lane, both halves of each 16-value step)
  uint32_t qa[8][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q + (size_t)lr * a.Hq * kD);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = 8 * ks + q;   // word index of dims 16 ks + 2q, +1
      qa[ks][0] = g < a.Hq ? q32[g * 64 + c] : 0u;
      qa[ks][1] = g + 8 < a.Hq ? q32[(g + 8) * 64 + c] : 0u;
      qa[ks][2] = g < a.Hq ? q32[g * 64 + c + 4] : 0u;
      qa[ks][3] = g + 8 < a.Hq ? q32[(g + 8) * 64 + c + 4] : 0u;
    }
  }
  uint8_t* buf0 = sm + (size_t)warp * 2 * kBufBytes;
  // stage group gi into buffer b: lane pair (2 lanes per token row half...) 16 tokens x 16
  // chunks of keys and of values, 8 copies per lane each
  auto stage = [&](int gi, int b) {
    uint8_t* kb = buf0 + b * kBufBytes;
    uint8_t* vb = kb + kGroup * kPitch;
    const uint32_t ka = smem_u32(kb), va = smem_u32(vb);
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int idx = it * 32 + lane;          // 0 .. 255: token idx >> 4, chunk idx & 15
      const int tk = idx >> 4, ch = idx & 15;
      const int j = gi * per_group + tk / a.bs;
      int blk = j < a.K ? sel[j] : -1;
      const bool ok = blk >= 0 && blk < nblk;
      const size_t t = ok ? (size_t)blk * a.bs + tk % a.bs : 0;
      cp_async16(ka + tk * kPitch + ch * 16, kl + t * 256 + ch * 16, ok);
      cp_async16(va + tk * kPitch + ch * 16, vl + t * 256 + ch * 16, ok);
    }
    cp_async_commit();
  };
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;   // heads g, g + 8
  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  const float scale = 0.08838834764831845f;   // 1 / sqrt(128) (fp32)
  int b = 0;
  int gi = gb + warp;
  if (gi < ge) stage(gi, 0);
  for (; gi < ge; gi += kWarps) {
    const int gn = gi + kWarps;
    if (gn < ge) stage(gn, b ^ 1);
    if (gn < ge) cp_async_wait<1>(); else cp_async_wait<0>();
    __syncwarp();
    const uint8_t* kb = buf0 + b * kBufBytes;
    const uint8_t* vb = kb + kGroup * kPitch;
    // which tokens of the group exist
    unsigned valid = 0u;
    {
      const int j = gi * per_group + (lane & 15) / a.bs;
      const int blk = (lane < 16 && j < a.K) ? sel[j] : -1;
      valid = __ballot_sync(0xffffffffu, lane < 16 && blk >= 0 && blk < nblk) & 0xFFFFu;
    }
    // S = Q K^T for tokens 0-7 (s[0]) and 8-15 (s[1])
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {   // two 16-value steps per ldmatrix.x4
        uint32_t r[4];
        // matrices: tokens 8nt..8nt+7 x dims 32kk + {0, 8, 16, 24} .. +7
        const int row = 8 * nt + (lane & 7), col = 32 * kk + 8 * (lane >> 3);
        ldsm_x4(smem_u32(kb + row * kPitch + col * 2), r);
        mma16816(s[nt], qa[2 * kk][0], qa[2 * kk][1], qa[2 * kk][2], qa[2 * kk][3], r[0], r[1]);
        mma16816(s[nt], qa[2 * kk + 1][0], qa[2 * kk + 1][1], qa[2 * kk + 1][2],
                 qa[2 * kk + 1][3], r[2], r[3]);
      }
    }
    // scale, mask, online softmax (this lane: heads g (s[.][0,1]) and g+8 (s[.][2,3]),
    // tokens 8 nt + 2q, 8 nt + 2q + 1)
    float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * nt + 2 * q + e;
        const bool on = (valid >> t) & 1u;
        s[nt][e] = on ? s[nt][e] * scale : kNegInf;
        s[nt][2 + e] = on ? s[nt][2 + e] * scale : kNegInf;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float c0 = n0 == kNegInf ? 1.f : expf(m0 - n0);
    const float c1 = n1 == kNegInf ? 1.f : expf(m1 - n1);
    float p[2][4];
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[nt][e] = s[nt][e] == kNegInf ? 0.f : expf(s[nt][e] - n0);
        p[nt][2 + e] = s[nt][2 + e] == kNegInf ? 0.f : expf(s[nt][2 + e] - n1);
        ps0 += p[nt][e];
        ps1 += p[nt][2 + e];
      }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      ps0 += __shfl_xor_sync(0xffffffffu, ps0, off);
      ps1 += __shfl_xor_sync(0xffffffffu, ps1, off);
    }
    l0 = l0 * c0 + ps0;
    l1 = l1 * c1 + ps1;
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= c0;
      o[nt][1] *= c0;
      o[nt][2] *= c1;
      o[nt][3] *= c1;
    }
    // P as the A operand (heads x 16 tokens), high and low bf16 parts
    uint32_t ph[4], pl[4];
    split_pair(p[0][0], p[0][1], &ph[0], &pl[0]);   // head g, tokens 2q, 2q+1
    split_pair(p[0][2], p[0][3], &ph[1], &pl[1]);   // head g+8
    split_pair(p[1][0], p[1][1], &ph[2], &pl[2]);   // head g, tokens 8+2q, 8+2q+1
    split_pair(p[1][2], p[1][3], &ph[3], &pl[3]);
    // O += P V over 16 dim tiles of 8 (V^T fragments by transposed ldmatrix)
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {   // two dim tiles per ldmatrix.x4
      uint32_t r[4];
      // matrices: tokens {0-7, 8-15} x dims 16dp + {0, 8}
      const int row = (lane & 7) + 8 * ((lane >> 3) & 1), col = 16 * dp + 8 * (lane >> 4);
      ldsm_x4_t(smem_u32(vb + row * kPitch + col * 2), r);
      mma16816(o[2 * dp], ph[0], ph[1], ph[2], ph[3], r[0], r[1]);
      mma16816(o[2 * dp], pl[0], pl[1], pl[2], pl[3], r[0], r[1]);
      mma16816(o[2 * dp + 1], ph[0], ph[1], ph[2], ph[3], r[2], r[3]);
      mma16816(o[2 * dp + 1], pl[0], pl[1], pl[2], pl[3], r[2], r[3]);
    }
    __syncwarp();   // the buffer is free for the group after next
    b ^= 1;
  }
  cp_async_wait<0>();
  __syncthreads();
  // merge the warps' states in warp order (shared memory reused), then this split's state
  // into the workspace
  float* ws = reinterpret_cast<float*>(sm);           // [warps][16 heads][130]
  {
    float* w = ws + (size_t)warp * 16 * 130;
    if (q == 0) {
      w[g * 130 + 0] = m0;
      w[g * 130 + 1] = l0;
      w[(g + 8) * 130 + 0] = m1;
      w[(g + 8) * 130 + 1] = l1;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      w[g * 130 + 2 + 8 * nt + 2 * q] = o[nt][0];
      w[g * 130 + 2 + 8 * nt + 2 * q + 1] = o[nt][1];
      w[(g + 8) * 130 + 2 + 8 * nt + 2 * q] = o[nt][2];
      w[(g + 8) * 130 + 2 + 8 * nt + 2 * q + 1] = o[nt][3];
    }
  }
  __syncthreads();
  float* part = a.part + ((size_t)sp * a.L * a.R + lr) * 16 * 130;
  for (int h = warp; h < 16; h += kWarps) {
    float M = kNegInf;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ws[((size_t)w * 16 + h) * 130]);
    float Lsum = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int w = 0; w < kWarps; ++w) {
      const float* src = ws + ((size_t)w * 16 + h) * 130;
      const float f = src[0] == kNegInf ? 0.f : expf(src[0] - M);
      Lsum += src[1] * f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] += src[2 + 32 * e + lane] * f;
    }
    if (lane == 0) {
      part[h * 130 + 0] = M;
      part[h * 130 + 1] = Lsum;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) part[h * 130 + 2 + 32 * e + lane] = acc[e];
  }
  // the CTA that finishes the row last merges the splits in split order and writes o
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.count[lr], 1) == a.splits - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int h = warp; h < a.Hq; h += kWarps) {
    float M = kNegInf;
    for (int x = 0; x < a.splits; ++x)
      M = fmaxf(M, __ldcg(a.part + (((size_t)x * a.L * a.R + lr) * 16 + h) * 130));
    float Lsum = 0.f;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int x = 0; x < a.splits; ++x) {
      const float* src = a.part + (((size_t)x * a.L * a.R + lr) * 16 + h) * 130;
      const float mx = __ldcg(src);
      const float f = mx == kNegInf ? 0.f : expf(mx - M);
      Lsum += __ldcg(src + 1) * f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] += __ldcg(src + 2 + 32 * e + lane) * f;
    }
    uint16_t* out = a.out + ((size_t)lr * a.Hq + h) * kD;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float val = Lsum > 0.f ? acc[e] / Lsum : 0.f;
      out[32 * e + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
    }
  }
  if (tid == 0) a.count[lr] = 0;   // ready for the next call on this workspace
}

}  // namespace

AttnLayout attn_layout(int L, int R, int splits) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  AttnLayout Ly{};
  size_t off = 0;
  Ly.header = off; off += 256;
  Ly.count = off; off += up(sizeof(int32_t) * (size_t)L * R);
  Ly.part = off; off += up(sizeof(float) * (size_t)splits * L * R * 16 * 130);
  Ly.total = off;
  return Ly;
}

int attn_splits(int L, int R) {
  // about four CTAs per SM in all, at most 8 per row
  const int rows = L * R;
  int s = (4 * device_sm_count() + rows - 1) / rows;
  return s < 1 ? 1 : (s > 8 ? 8 : s);
}

cudaError_t launch_attn(const AttnProblem& p, uint8_t* ws, cudaStream_t s) {
  const int splits = attn_splits(p.L, p.R);
  const AttnLayout Ly = attn_layout(p.L, p.R, splits);
  AttnArgs a{p.L, p.R, p.Hq, p.N, p.bs, p.K, p.kv_stride, p.q, p.k, p.v, p.sel, p.out,
             reinterpret_cast<float*>(ws + Ly.part), reinterpret_cast<int32_t*>(ws + Ly.count),
             reinterpret_cast<uint32_t*>(ws + Ly.header), splits};
  cudaError_t err =
      cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  k_attn<<<dim3(splits, p.L * p.R), kThreads, kSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsmoe
