// accept.cu — the acceptance step after a speculative verify: which drafted tokens are
// kept, and the one token the target model adds.
//
// Page: "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)",
// paragraph "DSpark": with the drafter on, a decode step verifies a block of 6 rows (the
// last committed token and 5 drafts) in one pass; under greedy decode the output is the
// same as without the drafter, and at temperature > 0 the step does exact speculative
// sampling. Row r's logits predict the token after row r's input, so draft r is checked
// against row r.
//
//  * Greedy: the argmax of every row (ties to the lowest token id); drafts are kept while
//    they equal the argmax of their row; the first mismatching row (or the last row)
//    adds its argmax.
//  * Sampling at temperature T: p_r = softmax(z_r / T) in fp64; draft d of row r is kept
//    iff u_acc[r] * q_r[d] < p_r[d] (q_r the drafter's distribution), i.e. with
//    probability min(1, p_r[d] / q_r[d]); at the first rejection the added token is drawn
//    from the residual max(p_r - q_r, 0) (from p_r if rounding leaves it empty) with
//    u_res[r]; after every draft is kept the bonus token is drawn from p_{R-1} with
//    u_res[R-1]. Drawing with u from weights w takes the smallest x whose cumulative
//    weight (token order) exceeds u * sum(w), else the last x with w[x] > 0.
//
// Every decision is taken in fp64 (on GB300 the fp64 exponentials of the softmax are the
// cost of sampling). The rows are split into chunks of kAcceptChunk tokens (kAcceptChunkSmall
// for small batches) over the GPU:
//   K_stats   per (chunk, row): greedy: the chunk's (max, lowest id); sampling: the
//             chunk's max m_c and sum_v exp(z_v / T - m_c / T).
//   K_decide  per step: each row's max M and normaliser s = sum_c s_c exp(m_c/T - M)
//             (chunks in order), then the rows' decisions in order.
//   K_part    per (chunk, step), sampling only: the chunk's residual and target weight
//             sums and last positive tokens for the row the step draws from.
//   K_pick    per step, sampling only: the chunk where the cumulative weight crosses
//             u * total, then the token inside it by a block scan.
#include "common.cuh"
#include "kernels.h"

namespace dsmoe {
namespace {

constexpr int kThreads = 256;
constexpr int kModeResidual = 0;                // draw from max(p - q, 0)
constexpr int kModeTarget = 1;                  // draw from p (bonus token)

struct AcceptArgs {
  const float* z;         // [B][R][V] logits
  int B, R, V, C;         // steps, rows, vocabulary, chunks per row
  double T;               // temperature (sampling)
  const double* qd;       // [B][R-1][V] drafter distributions (sampling)
  const int32_t* draft;   // [B][R-1]
  const double* u_acc;    // [B][R-1]
  const double* u_res;    // [B][R]
  int32_t* out;           // [B][R]
  int32_t* n_out;         // [B]
  AcceptChunk* cstat;     // [B][R][C]
  AcceptDecision* dec;    // [B]
  AcceptPart* spart;      // [B][C]
  uint32_t* status;
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide fp64 sum over kThreads threads (fixed tree order); every thread gets it.
__device__ double block_sum_d(double v, double* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double t = lane < kThreads / 32 ? sh[lane] : 0.0;
  t = warp_sum_d(t);
  __syncthreads();
  return t;
}

// (value, id) with the larger value, the lower id among equal values.
__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// ---------------------------------------------------------------------------------
// K_stats: one CTA per (chunk, row of a step); thread t reads tokens t, t + 256, ... of
// the chunk (coalesced), in ascending order.
// ---------------------------------------------------------------------------------
template <bool kGreedy, int CH>
__global__ void __launch_bounds__(kThreads) k_acc_stats(AcceptArgs a) {
  constexpr int kPer = CH / kThreads;   // tokens per thread in a chunk
  __shared__ double sh[32];
  __shared__ float shf[kThreads / 32];
  __shared__ int shi[kThreads / 32];
  const int c = blockIdx.x, br = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* z = a.z + (size_t)br * a.V;
  const int v0 = c * CH, v1 = min(a.V, v0 + CH);
  pdl_trigger();
  float best = -INFINITY;
  int bid = 0x7FFFFFFF;
  float zv[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int v = v0 + k * kThreads + (int)threadIdx.x;
    zv[k] = v < v1 ? __ldg(z + v) : -INFINITY;
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int v = v0 + k * kThreads + (int)threadIdx.x;
    if (v < v1) better(best, bid, zv[k], v);
  }
  // block (max, lowest id)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
    better(best, bid, ov, oi);
  }
  if (lane == 0) { shf[warp] = best; shi[warp] = bid; }
  __syncthreads();
  if (warp == 0) {
    best = lane < kThreads / 32 ? shf[lane] : -INFINITY;
    bid = lane < kThreads / 32 ? shi[lane] : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
      better(best, bid, ov, oi);
    }
    if (lane == 0) { shf[0] = best; shi[0] = bid; }
  }
  __syncthreads();
  AcceptChunk* cs = a.cstat + (size_t)br * a.C + c;
  if constexpr (kGreedy) {
    if (threadIdx.x == 0) {
      cs->m = shf[0];
      cs->id = shi[0];
      cs->s = 0.0;
    }
    return;
  }
  // sum of exp(z / T - m_c / T) over the chunk, in fp64 (z / T as z times 1 / T: within
  // an ulp of the quotient, far inside the decisions' rounding margin, and no fp64
  // division per token)
  const double invT = 1.0 / a.T;
  const double Mc = (double)shf[0] * invT;
  double s = 0.0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int v = v0 + k * kThreads + (int)threadIdx.x;
    if (v < v1) s += exp(fma((double)zv[k], invT, -Mc));
  }
  s = block_sum_d(s, sh);
  if (threadIdx.x == 0) {
    cs->m = shf[0];
    cs->id = shi[0];
    cs->s = s;
  }
}

// ---------------------------------------------------------------------------------
// K_decide: one warp per step. Each row's chunk results are combined lane-strided and
// then by a fixed shuffle tree; lane 0 takes the decisions in row order.
// ---------------------------------------------------------------------------------
template <bool kGreedy>
__global__ void __launch_bounds__(32) k_acc_decide(AcceptArgs a) {
  __shared__ double sM[kAcceptMaxRows], sS[kAcceptMaxRows];
  __shared__ int sBest[kAcceptMaxRows];
  const int b = blockIdx.x, lane = threadIdx.x;
  const int R = a.R, C = a.C;
  pdl_wait();   // the chunk results are complete
  pdl_trigger();
  for (int r = 0; r < R; ++r) {
    const AcceptChunk* cs = a.cstat + ((size_t)b * R + r) * C;
    if constexpr (kGreedy) {
      float best = -INFINITY;
      int bid = 0x7FFFFFFF;
      for (int c = lane; c < C; c += 32) better(best, bid, cs[c].m, cs[c].id);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
        better(best, bid, ov, oi);
      }
      if (lane == 0) sBest[r] = bid;
    } else {
      const double invT = 1.0 / a.T;   // z / T as z times 1 / T, as in the other kernels
      double M = -INFINITY;
      for (int c = lane; c < C; c += 32) M = fmax(M, (double)cs[c].m * invT);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmax(M, __shfl_xor_sync(0xffffffffu, M, o));
      double s = 0.0;
      for (int c = lane; c < C; c += 32) s += cs[c].s * exp(fma((double)cs[c].m, invT, -M));
      s = warp_sum_d(s);
      if (lane == 0) { sM[r] = M; sS[r] = s; }
    }
  }
  __syncwarp();
  if (lane != 0) return;
  int32_t* out = a.out + (size_t)b * R;
  int n = 0;
  if constexpr (kGreedy) {
    for (int r = 0; r < R; ++r) {
      out[n++] = sBest[r];
      if (r == R - 1 || a.draft[(size_t)b * (R - 1) + r] != sBest[r]) break;
    }
    for (int j = n; j < R; ++j) out[j] = -1;
    a.n_out[b] = n;
  } else {
    int rstar = R - 1, mode = kModeTarget;
    for (int r = 0; r < R - 1; ++r) {
      const int d = a.draft[(size_t)b * (R - 1) + r];
      bool keep = false;
      if (d >= 0 && d < a.V) {
        const double pd =
            exp(fma((double)a.z[((size_t)b * R + r) * a.V + d], 1.0 / a.T, -sM[r])) / sS[r];
        const double qv = a.qd[((size_t)b * (R - 1) + r) * a.V + d];
        keep = a.u_acc[(size_t)b * (R - 1) + r] * qv < pd;
      } else {
        flag_status(a.status, kStatusCheck);   // a draft outside the vocabulary: rejected
      }
      if (keep) {
        out[n++] = d;
        continue;
      }
      rstar = r;
      mode = kModeResidual;
      break;
    }
    for (int j = n; j < R; ++j) out[j] = -1;
    a.n_out[b] = n;   // the drawn token is appended by K_pick
    AcceptDecision& D = a.dec[b];
    D.row = rstar;
    D.mode = mode;
    D.M = sM[rstar];
    D.s = sS[rstar];
  }
}

// The target weight p_v and the residual weight max(p_v - q_v, 0) of token v.
// invT = 1 / T and inv_s = 1 / D.s are formed once per thread: a product within an ulp of
// the quotient, far inside the decisions' rounding margin.
__device__ __forceinline__ void weights(const AcceptDecision& D, double invT, double inv_s,
                                        const float* z, const double* q, int v, double* p,
                                        double* res) {
  *p = exp(fma((double)z[v], invT, -D.M)) * inv_s;
  if (D.mode == kModeResidual) {
    const double qv = q[v];
    *res = *p > qv ? *p - qv : 0.0;
  } else {
    *res = 0.0;
  }
}

// ---------------------------------------------------------------------------------
// K_part: one CTA per (chunk, step): sums of both weights over the chunk and the last
// token of the chunk with a positive weight of each kind.
// ---------------------------------------------------------------------------------
template <int CH>
__global__ void __launch_bounds__(kThreads) k_acc_part(AcceptArgs a) {
  constexpr int kPer = CH / kThreads;
  __shared__ double sh[32];
  __shared__ int shl[2];
  const int c = blockIdx.x, b = blockIdx.y;
  pdl_wait();   // the decisions are complete
  pdl_trigger();
  const AcceptDecision D = a.dec[b];
  const double invT = 1.0 / a.T, inv_s = 1.0 / D.s;
  const float* z = a.z + ((size_t)b * a.R + D.row) * a.V;
  const double* q =
      D.mode == kModeResidual ? a.qd + ((size_t)b * (a.R - 1) + D.row) * a.V : nullptr;
  const int v0 = c * CH, v1 = min(a.V, v0 + CH);
  if (threadIdx.x == 0) { shl[0] = -1; shl[1] = -1; }
  __syncthreads();
  double sp = 0.0, sr = 0.0;
  int lp = -1, lr = -1;
  for (int k = 0; k < kPer; ++k) {
    const int v = v0 + k * kThreads + (int)threadIdx.x;
    if (v < v1) {
      double p, r;
      weights(D, invT, inv_s, z, q, v, &p, &r);
      sp += p;
      sr += r;
      if (p > 0.0) lp = v;
      if (r > 0.0) lr = v;
    }
  }
  if (lp >= 0) atomicMax(&shl[1], lp);
  if (lr >= 0) atomicMax(&shl[0], lr);
  sp = block_sum_d(sp, sh);
  sr = block_sum_d(sr, sh);
  if (threadIdx.x == 0) {
    AcceptPart& P = a.spart[(size_t)b * a.C + c];
    P.res = sr;
    P.p = sp;
    P.last_res = shl[0];
    P.last_p = shl[1];
  }
}

// ---------------------------------------------------------------------------------
// K_pick: one CTA per step. The chunk sums are added in chunk order to find the chunk in
// which the cumulative weight first exceeds u * total; inside it, thread t takes kPer
// consecutive tokens (sequential partial sums) and a block scan of the threads' totals
// gives every token's cumulative weight; the smallest token past the target is drawn.
// ---------------------------------------------------------------------------------
template <int CH>
__global__ void __launch_bounds__(kThreads) k_acc_pick(AcceptArgs a) {
  constexpr int kPer = CH / kThreads;
  __shared__ double sh[kThreads / 32];
  __shared__ int s_chunk, s_tok, s_use_res, s_last;
  __shared__ double s_target, s_pre;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();   // the chunk sums are complete
  const AcceptDecision D = a.dec[b];
  const AcceptPart* P = a.spart + (size_t)b * a.C;
  if (tid == 0) {
    double tres = 0.0, tp = 0.0;
    int last_res = -1, last_p = -1;
    for (int c = 0; c < a.C; ++c) {
      tres += P[c].res;
      tp += P[c].p;
      last_res = max(last_res, P[c].last_res);
      last_p = max(last_p, P[c].last_p);
    }
    const bool use_res = D.mode == kModeResidual && tres > 0.0;
    const double total = use_res ? tres : tp;
    const double target = a.u_res[(size_t)b * a.R + D.row] * total;
    int chunk = -1;
    double pre = 0.0;
    for (int c = 0; c < a.C; ++c) {
      const double w = use_res ? P[c].res : P[c].p;
      if (target < pre + w) { chunk = c; break; }
      pre += w;
    }
    s_use_res = use_res ? 1 : 0;
    s_chunk = chunk;
    s_target = target;
    s_pre = pre;
    s_tok = chunk < 0 ? (use_res ? last_res : last_p) : 0x7FFFFFFF;
  }
  __syncthreads();
  if (s_chunk >= 0) {
    const int c = s_chunk;
    const double invT = 1.0 / a.T, inv_s = 1.0 / D.s;
    const float* z = a.z + ((size_t)b * a.R + D.row) * a.V;
    const double* q =
        D.mode == kModeResidual ? a.qd + ((size_t)b * (a.R - 1) + D.row) * a.V : nullptr;
    const int v0 = c * CH + tid * kPer, v1 = min(a.V, c * CH + CH);
    double w[kPer];
    double mine = 0.0;
    for (int k = 0; k < kPer; ++k) {
      const int v = v0 + k;
      double p = 0.0, r = 0.0;
      if (v < v1) weights(D, invT, inv_s, z, q, v, &p, &r);
      w[k] = s_use_res ? r : p;
      mine += w[k];
    }
    // exclusive scan of the threads' totals (warp scans, then the warps' totals)
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    double wpre = 0.0;
    for (int j = 0; j < warp; ++j) wpre += sh[j];
    double acc = s_pre + wpre + (incl - mine);
    int tok = 0x7FFFFFFF, last_pos = -1;
    for (int k = 0; k < kPer; ++k) {
      const int v = v0 + k;
      if (v >= v1) break;
      acc += w[k];
      if (w[k] > 0.0) last_pos = v;
      if (s_target < acc) { tok = v; break; }
    }
    __syncthreads();
    if (tid == 0) { s_tok = 0x7FFFFFFF; s_last = -1; }
    __syncthreads();
    atomicMin(&s_tok, tok);
    if (last_pos >= 0) atomicMax(&s_last, last_pos);
    __syncthreads();
    // none inside the chunk (the scan's rounding): the chunk's last positive token
    if (tid == 0 && s_tok == 0x7FFFFFFF) s_tok = s_last;
  }
  __syncthreads();
  if (tid == 0) {
    const int n = a.n_out[b];
    a.out[(size_t)b * a.R + n] = s_tok;
    a.n_out[b] = n + 1;
  }
}

}  // namespace

AcceptLayout accept_layout(int B, int R, int V) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  // sized for the smaller chunk
  const size_t C = (size_t)(V + kAcceptChunkSmall - 1) / kAcceptChunkSmall;
  AcceptLayout L{};
  size_t off = 0;
  L.header = off; off += 256;
  L.cstat = off; off += up(sizeof(AcceptChunk) * (size_t)B * R * C);
  L.dec = off; off += up(sizeof(AcceptDecision) * (size_t)B);
  L.spart = off; off += up(sizeof(AcceptPart) * (size_t)B * C);
  L.total = off;
  return L;
}

template <int CH>
cudaError_t launch_accept_ch(AcceptArgs a, bool greedy, cudaStream_t s) {
  a.C = (a.V + CH - 1) / CH;
  const dim3 g1(a.C, a.B * a.R);
  if (greedy) {
    k_acc_stats<true, CH><<<g1, kThreads, 0, s>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_pdl(k_acc_decide<true>, a.B, 32, 0, s, a);
  }
  k_acc_stats<false, CH><<<g1, kThreads, 0, s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if ((err = launch_pdl(k_acc_decide<false>, a.B, 32, 0, s, a)) != cudaSuccess) return err;
  if ((err = launch_pdl(k_acc_part<CH>, dim3(a.C, a.B), kThreads, 0, s, a)) != cudaSuccess)
    return err;
  return launch_pdl(k_acc_pick<CH>, a.B, kThreads, 0, s, a);
}

cudaError_t launch_accept(const AcceptProblem& pr, uint8_t* ws, cudaStream_t s) {
  const AcceptLayout L = accept_layout(pr.B, pr.R, pr.V);
  AcceptArgs a{};
  a.z = pr.logits;
  a.B = pr.B; a.R = pr.R; a.V = pr.V;
  a.T = pr.T;
  a.qd = pr.qd; a.draft = pr.draft; a.u_acc = pr.u_acc; a.u_res = pr.u_res;
  a.out = pr.out; a.n_out = pr.n_out;
  a.cstat = reinterpret_cast<AcceptChunk*>(ws + L.cstat);
  a.dec = reinterpret_cast<AcceptDecision*>(ws + L.dec);
  a.spart = reinterpret_cast<AcceptPart*>(ws + L.spart);
  a.status = reinterpret_cast<uint32_t*>(ws + L.header);
  // Chunks of kAcceptChunk tokens, or of kAcceptChunkSmall when that leaves fewer than
  // two CTAs per SM (few steps): the later kernels work on one row per step and the draw
  // scans one chunk, so small batches want short chunks.
  const long long ctas = (long long)pr.B * pr.R * ((pr.V + kAcceptChunk - 1) / kAcceptChunk);
  if (ctas < 2LL * device_sm_count()) return launch_accept_ch<kAcceptChunkSmall>(a, pr.greedy, s);
  return launch_accept_ch<kAcceptChunk>(a, pr.greedy, s);
}

}  // namespace dsmoe
