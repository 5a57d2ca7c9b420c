// kernels.h — internal interface between the host API (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>   // CUtensorMap
#include <cuda_runtime.h>

#include "dsmoe.h"

namespace dsmoe {

constexpr int kMaxRows = 6;        // verify rows per MoE call
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kMaxUnion = kMaxRows * kMaxTopK;

// Routing result shared by K1 (writer) and K3/K4 (readers); lives in the workspace.
struct RouteInfo {
  int32_t n_union;                  // distinct routed experts over the R rows
  int32_t pad[3];
  int32_t expert[kMaxUnion];        // ascending expert id
  uint32_t rowmask[kMaxUnion];      // bit r: row r selected this expert
  int8_t slot[kMaxUnion][8];        // rank + 1 of the expert in row r (slot 0 = shared)
};

struct MoeDims {
  int R, H, E, I, k;
};

// Bytes of one tile of the tile-major Q4 layout: 16 rows x 64 values, 512 bytes of nibbles
// in tensor-core fragment order followed by 64 bytes of fp16 scales.
constexpr int kQ4TileBytes = 576;

struct MoeWorkspace {
  uint32_t* header;        // status word, arrival counts and flags (zeroed per call)
  size_t zero_bytes;       // bytes from header on that every call zeroes first
  float* scores;           // [R][E] sigmoid router scores
  RouteInfo* route;
  uint16_t* h;             // bf16 [R][1+k][I]
  float* opart;            // [R][1+k][H] expert outputs before the combine
};

struct MoeLayout {
  size_t header, scores, route, h, opart, total, zero_bytes;
};
MoeLayout moe_layout(const MoeDims& d);
// The layer's kernel fits this device's shared memory (the R verify rows are staged there).
bool moe_fits(const MoeDims& d);

// n_mats planar Q4 matrices (qs [rows][K/2], sc [rows][K/32] each) -> tile-major with
// tile rows in groups of `group` (rows % 16 == 0, K % 64 == 0).
cudaError_t launch_tile(const uint8_t* qs, const uint16_t* sc, int n_mats, int64_t rows,
                        int K, int group, uint8_t* dst, cudaStream_t s);
// Tile rows per group of the down-projection matrices (gate and up use groups of 1).
constexpr int kDownGroup = DS_Q4_DOWN_GROUP;
// The whole verify step of one layer: a prologue that zeroes the workspace header (then
// `after_prologue` is recorded when not null), and one cooperative kernel (router,
// gate/up/SwiGLU, down projection, combine).
cudaError_t launch_moe(const MoeDims& d, const uint16_t* x, const uint16_t* router_w,
                       const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                       const uint8_t* sh_gate, const uint8_t* sh_up, const uint8_t* sh_down,
                       int32_t* topk_idx, float* topk_w, uint16_t* y, const MoeWorkspace& ws,
                       cudaStream_t s, cudaEvent_t after_prologue);

// ------------------------------------------------------------------ block select ----
struct SelDims {
  int L, R, Hh, D, N, topk;
  int64_t key_stride;
};

struct SelWorkspace {
  uint32_t* header;
  uint32_t* ldone;    // [L] rows of the layer whose top-k is done (zeroed with the header)
  uint32_t* uagg;     // [L][P] union count of each chunk of kCompactChunk mask words, with
                      // bit 31 set once published (zeroed with the header by every call)
  int32_t* wordoff;   // [L][W] exclusive prefix of union-admitted counts per mask word
  int32_t* cidx;      // [L][R][N] (caller's array or workspace)
  int32_t* ccount;    // [L][R]
  int32_t* uidx;      // [L][N] union of the rows' admitted blocks, ascending
  int32_t* ucount;    // [L]
  uint8_t* urows;     // [L][N] bit r: row r admits the union entry
  float* cscore;      // [L][R][NS] by union entry: canonical or tensor-core scores
                      // (-inf where the row does not admit the entry)
  float* knorm;       // [L][NS] by union entry: key norm bound (tensor-core scoring)
  float* kmax;        // [L][NC] the largest knorm of each 32 union entries (NC = NS / 32
                      // rounded up; tensor-core scoring)
  float* qnorm;       // [L][R] sum_h |w_h| ||q_h|| bound (tensor-core scoring)
  float* smax;        // [L][NC][R] per 32 union entries, the largest score each row gives
                      // them (-inf: none admitted; tensor-core scoring)
};

// Row stride of the score arrays (cscore, knorm): N rounded up to a multiple of 32, so that
// every row starts on a 128-byte line (rows are dropped from L2 line by line once read).
inline int score_stride(int N) { return (N + 31) & ~31; }
// Row stride of kmax: one value per 32 union entries.
inline int chunk_stride(int N) { return (score_stride(N) + 31) / 32; }

struct SelLayout {
  size_t header, uagg, ldone, zero_bytes, wordoff, cidx, ccount, uidx, ucount, urows, cscore, knorm,
      kmax, qnorm, smax, total;
};
SelLayout sel_layout(const SelDims& d, bool caller_cidx);
bool tc_scoring_supported(const SelDims& d, const uint16_t* keys, const uint16_t* q);

cudaError_t launch_compact(const SelDims& d, const uint32_t* mask, const int32_t* limit,
                           const SelWorkspace& ws, bool want_cidx, cudaStream_t s);
cudaError_t launch_score(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                         const float* head_w, const uint32_t* mask, const int32_t* limit,
                         const SelWorkspace& ws, bool tc, cudaStream_t s);
cudaError_t launch_topk(const SelDims& d, const uint16_t* keys, const uint16_t* q,
                        const float* head_w, int32_t* sel, int32_t* nsel,
                        const SelWorkspace& ws, bool tc, bool keep, cudaStream_t s);

// TMA tensor map (cached by its parameters) of bf16 block keys [L][N][128] (layer stride
// key_stride values, a multiple of 8) in boxes of 64 values x box_rows blocks, 128-byte
// swizzle.
cudaError_t key_tile_map(CUtensorMap* out, const uint16_t* keys, int N, int L,
                         int64_t key_stride, int box_rows);

// ---- paired Q8 projections (q8.cu)
constexpr int kQ8TileBytes = 1088;   // 16 rows x 64 int8 values + 32 fp16 scales
constexpr int kQ8MaxStages = 16;
constexpr int kQ8MaxSlots = 40;
size_t q8_tiled_bytes(long long rows, int K);
cudaError_t launch_q8_tile(const int8_t* qs, const uint16_t* sc, int rows, int K, void* dst,
                           cudaStream_t s);
bool q8_plan(int R, int K, int* stages, int* slots, size_t* smem);
cudaError_t launch_q8_project(const void* tiles, int rows, int K, const uint16_t* x, int R,
                              uint16_t* y, uint32_t* status, cudaStream_t s);

// ---- sparse attention over the selected blocks (attn.cu)
struct AttnProblem {
  int L, R, Hq, N, bs, K;
  int64_t kv_stride;
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* sel;
  uint16_t* out;
};
struct AttnLayout {
  size_t header, count, part, total;
};
int attn_splits(int L, int R);
AttnLayout attn_layout(int L, int R, int splits);
cudaError_t launch_attn(const AttnProblem& p, uint8_t* ws, cudaStream_t s);

// ---- verify acceptance (accept.cu)
constexpr int kAcceptChunk = 4096;    // tokens of a row per CTA
constexpr int kAcceptChunkSmall = 1024;   // the same for batches of few steps
constexpr int kAcceptMaxRows = 16;
struct AcceptChunk {      // per (step, row, chunk)
  float m;                // greedy / sampling: the chunk's largest logit
  int32_t id;             // greedy: its lowest token id
  double s;               // sampling: sum of exp(z / T - m / T) over the chunk
};
struct AcceptDecision {   // per step (sampling)
  int32_t row, mode;      // the row the added token is drawn from; residual or target
  double M, s;            // that row's max logit / T and softmax normaliser
};
struct AcceptPart {       // per (step, chunk) (sampling)
  double res, p;          // residual and target weight sums of the chunk
  int32_t last_res, last_p;   // the chunk's last token with a positive weight (-1: none)
};
struct AcceptLayout {
  size_t header, cstat, dec, spart, total;
};
struct AcceptProblem {
  const float* logits;
  int B, R, V;
  bool greedy;
  double T;
  const double* qd;
  const int32_t* draft;
  const double* u_acc;
  const double* u_res;
  int32_t* out;
  int32_t* n_out;
};
AcceptLayout accept_layout(int B, int R, int V);
cudaError_t launch_accept(const AcceptProblem& p, uint8_t* ws, cudaStream_t s);

// Cached device properties of the current device.
int device_sm_count();
int device_max_smem_optin();

}  // namespace dsmoe
