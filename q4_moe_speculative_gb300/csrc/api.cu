// api.cu — the C ABI of libdsmoe.so: host-side validation, workspace carving and the
// launch sequence of each call. Nothing here allocates memory or synchronises, except
// ds_workspace_status(), which synchronises the stream to read the device status word.
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace dsmoe {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

int device_max_smem_optin() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      n = 48 * 1024;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace dsmoe

using namespace dsmoe;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool tiles_ok(const ds_q4_tiled& w) { return w.tiles && aligned(w.tiles, 16); }

// Sizes only (no pointers): DS_ERR_INVALID_ARG outside the format's limits (H and I
// multiples of 32, ranges, k, E, R), DS_ERR_UNSUPPORTED for valid sizes this build's
// kernels do not run (H or I not a multiple of 64).
ds_status check_layer_sizes(const ds_moe_layer* L, int32_t R) {
  if (!L) return DS_ERR_INVALID_ARG;
  if (R < 1 || R > kMaxRows) return DS_ERR_INVALID_ARG;
  if (L->hidden < 64 || L->hidden > 16384 || L->hidden % 32) return DS_ERR_INVALID_ARG;
  if (L->inter < 64 || L->inter > 8192 || L->inter % 32) return DS_ERR_INVALID_ARG;
  if (L->top_k < 1 || L->top_k > kMaxTopK) return DS_ERR_INVALID_ARG;
  if (L->n_experts < L->top_k || L->n_experts > kMaxExperts) return DS_ERR_INVALID_ARG;
  if (L->hidden % 64 || L->inter % 64) return DS_ERR_UNSUPPORTED;
  return DS_OK;
}

ds_status check_layer(const ds_moe_layer* L, int32_t R) {
  const ds_status st = check_layer_sizes(L, R);
  if (st != DS_OK) return st;
  if (!L->router_w || !aligned(L->router_w, 16)) return DS_ERR_INVALID_ARG;
  if (!tiles_ok(L->gate) || !tiles_ok(L->up) || !tiles_ok(L->down) || !tiles_ok(L->sh_gate) ||
      !tiles_ok(L->sh_up) || !tiles_ok(L->sh_down))
    return DS_ERR_INVALID_ARG;
  return DS_OK;
}

MoeDims dims_of(const ds_moe_layer* L, int32_t R) {
  return MoeDims{R, L->hidden, L->n_experts, L->inter, L->top_k};
}

ds_status check_select(const ds_select_args* a) {
  if (!a) return DS_ERR_INVALID_ARG;
  if (a->n_layers < 1 || a->n_rows < 1 || a->n_rows > 8) return DS_ERR_INVALID_ARG;
  if (a->n_heads < 1 || a->n_heads > 16 || a->head_dim != 128) return DS_ERR_INVALID_ARG;
  if (a->n_blocks < 1 || a->n_blocks > (1 << 24)) return DS_ERR_INVALID_ARG;
  if (a->top_k < 1 || a->top_k > 2048) return DS_ERR_INVALID_ARG;
  if (a->key_layer_stride < (int64_t)a->n_blocks * a->head_dim || a->key_layer_stride % 8)
    return DS_ERR_INVALID_ARG;
  if (!a->keys || !aligned(a->keys, 16) || !a->q || !aligned(a->q, 4) || !a->head_w ||
      !a->mask || !a->limit)
    return DS_ERR_INVALID_ARG;
  if (a->flags & ~(DS_SELECT_CANONICAL_SCORES | DS_SELECT_KEEP_WORKSPACE)) return DS_ERR_INVALID_ARG;
  return DS_OK;
}

// Records marks[i] on s when present; false if recording failed.
bool mark(const ds_event_t* marks, int i, cudaStream_t s) {
  if (!marks || !marks[i]) return true;
  return cudaEventRecord(reinterpret_cast<cudaEvent_t>(marks[i]), s) == cudaSuccess;
}

SelDims sdims_of(const ds_select_args* a) {
  return SelDims{a->n_layers, a->n_rows, a->n_heads, a->head_dim, a->n_blocks, a->top_k,
                 a->key_layer_stride};
}

}  // namespace

extern "C" {

size_t ds_q4_tiled_bytes(int64_t rows, int32_t K) {
  if (rows <= 0 || rows % 16 || K <= 0 || K % 64) return 0;
  return (size_t)rows / 16 * (size_t)(K / 64) * kQ4TileBytes;
}

ds_status ds_q4_tile(const ds_q4* src, int32_t n_mats, int64_t rows, int32_t K, int32_t group,
                     void* dst, size_t dst_bytes, ds_stream_t stream) {
  if (!src || !src->qs || !src->sc || !dst || !aligned(src->qs, 4) || !aligned(src->sc, 2) ||
      !aligned(dst, 16))
    return DS_ERR_INVALID_ARG;
  if (n_mats < 1 || group < 1 || group > 65536 || rows > ((int64_t)1 << 40)) return DS_ERR_INVALID_ARG;
  const size_t need = ds_q4_tiled_bytes(rows, K);
  if (need == 0) return DS_ERR_INVALID_ARG;
  if (dst_bytes / (size_t)n_mats < need) return DS_ERR_WORKSPACE;
  return launch_tile(src->qs, src->sc, n_mats, rows, K, group, static_cast<uint8_t*>(dst),
                     reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DS_OK
             : DS_ERR_CUDA;
}

size_t ds_moe_workspace_size(const ds_moe_layer* layer, int32_t R) {
  if (check_layer_sizes(layer, R) != DS_OK) return 0;
  return moe_layout(dims_of(layer, R)).total;
}

ds_status ds_moe_verify_forward(const ds_moe_layer* layer, const uint16_t* x, int32_t R,
                                uint16_t* y, int32_t* topk_idx, float* topk_w,
                                void* workspace, size_t ws_bytes, ds_stream_t stream) {
  return ds_moe_verify_forward_marked(layer, x, R, y, topk_idx, topk_w, workspace, ws_bytes,
                                      stream, nullptr);
}

ds_status ds_moe_verify_forward_marked(const ds_moe_layer* layer, const uint16_t* x,
                                       int32_t R, uint16_t* y, int32_t* topk_idx,
                                       float* topk_w, void* workspace, size_t ws_bytes,
                                       ds_stream_t stream, const ds_event_t marks[3]) {
  ds_status st = check_layer(layer, R);
  if (st != DS_OK) return st;
  if (!x || !y || !topk_idx || !topk_w || !aligned(x, 16) || !aligned(y, 4) ||
      !aligned(topk_idx, 4) || !aligned(topk_w, 4))
    return DS_ERR_INVALID_ARG;
  const MoeDims d = dims_of(layer, R);
  const MoeLayout L = moe_layout(d);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return DS_ERR_WORKSPACE;
  // The verify rows are staged in shared memory: R * (2H + 64) bytes beside the weight stages.
  if (!moe_fits(d)) return DS_ERR_UNSUPPORTED;

  char* base = static_cast<char*>(workspace);
  MoeWorkspace ws{};
  ws.header = reinterpret_cast<uint32_t*>(base + L.header);
  ws.zero_bytes = L.zero_bytes;
  ws.scores = reinterpret_cast<float*>(base + L.scores);
  ws.route = reinterpret_cast<RouteInfo*>(base + L.route);
  ws.h = reinterpret_cast<uint16_t*>(base + L.h);
  ws.opart = reinterpret_cast<float*>(base + L.opart);

  auto t = [](const ds_q4_tiled& m) { return static_cast<const uint8_t*>(m.tiles); };
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t m0 = (marks && marks[0]) ? reinterpret_cast<cudaEvent_t>(marks[0]) : nullptr;
  if (launch_moe(d, x, layer->router_w, t(layer->gate), t(layer->up), t(layer->down),
                 t(layer->sh_gate), t(layer->sh_up), t(layer->sh_down), topk_idx, topk_w, y, ws,
                 s, m0) != cudaSuccess)
    return DS_ERR_CUDA;
  if (!mark(marks, 1, s) || !mark(marks, 2, s)) return DS_ERR_CUDA;
  return DS_OK;
}

size_t ds_moe_workspace_h_offset(const ds_moe_layer* layer, int32_t R) {
  if (ds_moe_workspace_size(layer, R) == 0) return (size_t)-1;
  return moe_layout(dims_of(layer, R)).h;
}

size_t ds_select_workspace_size(const ds_select_args* args) {
  if (check_select(args) != DS_OK) return 0;
  // Sized for the case where the caller does not pass cidx / ccount.
  return sel_layout(sdims_of(args), false).total;
}

size_t ds_select_workspace_offset(const ds_select_args* args, int32_t with_compacted,
                                  int32_t part) {
  if (check_select(args) != DS_OK) return (size_t)-1;
  const SelLayout L = sel_layout(sdims_of(args), with_compacted != 0);
  switch (part) {
    case DS_SELECT_WS_UNION: return L.uidx;
    case DS_SELECT_WS_UNION_COUNT: return L.ucount;
    case DS_SELECT_WS_SCORES: return L.cscore;
    case DS_SELECT_WS_KEY_NORMS: return L.knorm;
    case DS_SELECT_WS_ROW_SCALES: return L.qnorm;
  }
  return (size_t)-1;
}

ds_status ds_select_blocks(const ds_select_args* a, int32_t* sel, int32_t* nsel, int32_t* cidx,
                           int32_t* ccount, void* workspace, size_t ws_bytes,
                           ds_stream_t stream) {
  return ds_select_blocks_marked(a, sel, nsel, cidx, ccount, workspace, ws_bytes, stream,
                                 nullptr);
}

ds_status ds_select_blocks_marked(const ds_select_args* a, int32_t* sel, int32_t* nsel,
                                  int32_t* cidx, int32_t* ccount, void* workspace,
                                  size_t ws_bytes, ds_stream_t stream,
                                  const ds_event_t marks[3]) {
  ds_status st = check_select(a);
  if (st != DS_OK) return st;
  if (!sel || !nsel || (cidx == nullptr) != (ccount == nullptr) || !aligned(sel, 4) ||
      !aligned(nsel, 4))
    return DS_ERR_INVALID_ARG;
  const SelDims d = sdims_of(a);
  const bool caller = cidx != nullptr;
  const SelLayout L = sel_layout(d, caller);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return DS_ERR_WORKSPACE;

  char* base = static_cast<char*>(workspace);
  SelWorkspace ws{};
  ws.header = reinterpret_cast<uint32_t*>(base + L.header);
  ws.uagg = reinterpret_cast<uint32_t*>(base + L.uagg);
  ws.ldone = reinterpret_cast<uint32_t*>(base + L.ldone);
  ws.wordoff = reinterpret_cast<int32_t*>(base + L.wordoff);
  ws.cidx = caller ? cidx : reinterpret_cast<int32_t*>(base + L.cidx);
  ws.ccount = caller ? ccount : reinterpret_cast<int32_t*>(base + L.ccount);
  ws.uidx = reinterpret_cast<int32_t*>(base + L.uidx);
  ws.ucount = reinterpret_cast<int32_t*>(base + L.ucount);
  ws.urows = reinterpret_cast<uint8_t*>(base + L.urows);
  ws.cscore = reinterpret_cast<float*>(base + L.cscore);
  ws.knorm = reinterpret_cast<float*>(base + L.knorm);
  ws.kmax = reinterpret_cast<float*>(base + L.kmax);
  ws.qnorm = reinterpret_cast<float*>(base + L.qnorm);
  ws.smax = reinterpret_cast<float*>(base + L.smax);
  const bool tc = !(a->flags & DS_SELECT_CANONICAL_SCORES) &&
                  tc_scoring_supported(d, a->keys, a->q);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(base, 0, L.zero_bytes, s) != cudaSuccess) return DS_ERR_CUDA;
  if (launch_compact(d, a->mask, a->limit, ws, caller, s) != cudaSuccess) return DS_ERR_CUDA;
  if (!mark(marks, 0, s)) return DS_ERR_CUDA;
  if (launch_score(d, a->keys, a->q, a->head_w, a->mask, a->limit, ws, tc, s) != cudaSuccess)
    return DS_ERR_CUDA;
  if (!mark(marks, 1, s)) return DS_ERR_CUDA;
  if (launch_topk(d, a->keys, a->q, a->head_w, sel, nsel, ws, tc,
                  (a->flags & DS_SELECT_KEEP_WORKSPACE) != 0, s) != cudaSuccess)
    return DS_ERR_CUDA;
  if (!mark(marks, 2, s)) return DS_ERR_CUDA;
  return DS_OK;
}

namespace {

ds_status check_attn(const ds_attn_args* a) {
  if (!a) return DS_ERR_INVALID_ARG;
  if (a->n_layers < 1 || a->n_rows < 1 || a->n_rows > 8 || a->n_heads < 1 || a->n_heads > 16)
    return DS_ERR_INVALID_ARG;
  const int bs = a->block_tokens;
  if (!(bs == 1 || bs == 2 || bs == 4 || bs == 8 || bs == 16)) return DS_ERR_INVALID_ARG;
  if (a->n_blocks < 1 || a->n_blocks > (1 << 24) || a->top_k < 1 || a->top_k > 2048)
    return DS_ERR_INVALID_ARG;
  if (a->head_dim < 1) return DS_ERR_INVALID_ARG;
  if (a->head_dim != 128) return DS_ERR_UNSUPPORTED;
  if ((long long)a->n_layers * a->n_rows > 65535) return DS_ERR_INVALID_ARG;
  if (a->kv_layer_stride < (int64_t)a->n_blocks * bs * a->head_dim) return DS_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || !a->sel) return DS_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->sel, 4))
    return DS_ERR_INVALID_ARG;
  if (a->kv_layer_stride % 8) return DS_ERR_INVALID_ARG;   // 16-byte aligned layers
  return DS_OK;
}

}  // namespace

size_t ds_attn_workspace_size(const ds_attn_args* a) {
  if (check_attn(a) != DS_OK) return 0;
  return attn_layout(a->n_layers, a->n_rows, attn_splits(a->n_layers, a->n_rows)).total;
}

ds_status ds_sparse_attention(const ds_attn_args* a, uint16_t* out, void* workspace,
                              size_t ws_bytes, ds_stream_t stream) {
  const ds_status st = check_attn(a);
  if (st != DS_OK) return st;
  if (!out || !aligned(out, 16)) return DS_ERR_INVALID_ARG;
  const int splits = attn_splits(a->n_layers, a->n_rows);
  const AttnLayout Ly = attn_layout(a->n_layers, a->n_rows, splits);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < Ly.total) return DS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  if (cudaMemsetAsync(base, 0, Ly.part, s) != cudaSuccess) return DS_ERR_CUDA;   // header, counts
  AttnProblem p{a->n_layers, a->n_rows, a->n_heads, a->n_blocks, a->block_tokens, a->top_k,
                a->kv_layer_stride, a->q, a->k, a->v, a->sel, out};
  return launch_attn(p, base, s) == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

namespace {

bool q8_sizes_ok(int64_t rows, int32_t K) {
  return rows >= 16 && rows <= (1 << 24) && rows % 16 == 0 && K >= 32 && K <= 65536 &&
         K % 32 == 0;
}

}  // namespace

size_t ds_q8_tiled_bytes(int64_t rows, int32_t K) {
  if (!q8_sizes_ok(rows, K) || K % 64) return 0;
  return q8_tiled_bytes(rows, K);
}

ds_status ds_q8_tile(const ds_q8* src, int64_t rows, int32_t K, void* dst, size_t dst_bytes,
                     ds_stream_t stream) {
  if (!src || !src->qs || !src->sc || !dst) return DS_ERR_INVALID_ARG;
  if (!q8_sizes_ok(rows, K) || K % 64) return DS_ERR_INVALID_ARG;
  if (!aligned(src->qs, 16) || !aligned(src->sc, 16) || !aligned(dst, 16))
    return DS_ERR_INVALID_ARG;
  if (dst_bytes < q8_tiled_bytes(rows, K)) return DS_ERR_WORKSPACE;
  return launch_q8_tile(src->qs, src->sc, (int)rows, K, dst,
                        reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DS_OK
             : DS_ERR_CUDA;
}

size_t ds_q8_workspace_size(void) { return 256; }

ds_status ds_q8_project(const ds_q8_tiled* w, int64_t rows, int32_t K, const uint16_t* x,
                        int32_t R, uint16_t* y, void* workspace, size_t ws_bytes,
                        ds_stream_t stream) {
  if (!w || !w->tiles || !x || !y) return DS_ERR_INVALID_ARG;
  if (!q8_sizes_ok(rows, K) || R < 1 || R > 8) return DS_ERR_INVALID_ARG;
  if (!aligned(w->tiles, 16) || !aligned(x, 16) || !aligned(y, 16)) return DS_ERR_INVALID_ARG;
  if (K % 1024) return DS_ERR_UNSUPPORTED;
  int S = 0, P = 0;
  size_t smem = 0;
  if (!q8_plan(R, K, &S, &P, &smem)) return DS_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 256) || ws_bytes < 256) return DS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // (the kernel resets the status word itself, so that consecutive projections overlap)
  return launch_q8_project(w->tiles, (int)rows, K, x, R, y, static_cast<uint32_t*>(workspace), s) ==
                 cudaSuccess
             ? DS_OK
             : DS_ERR_CUDA;
}

namespace {

bool verify_sizes_ok(int32_t B, int32_t R, int32_t V) {
  return B >= 1 && B <= 4096 && R >= 1 && R <= kAcceptMaxRows && V >= 1 && V <= (1 << 24);
}

ds_status verify_call(AcceptProblem& pr, void* workspace, size_t ws_bytes, ds_stream_t stream) {
  if (!pr.logits || !pr.out || !pr.n_out) return DS_ERR_INVALID_ARG;
  if (pr.R > 1 && !pr.draft) return DS_ERR_INVALID_ARG;
  const AcceptLayout L = accept_layout(pr.B, pr.R, pr.V);
  if (!workspace || !aligned(workspace, 256) || ws_bytes < L.total) return DS_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  if (cudaMemsetAsync(base, 0, 256, s) != cudaSuccess) return DS_ERR_CUDA;
  return launch_accept(pr, base, s) == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

}  // namespace

size_t ds_verify_workspace_size(int32_t B, int32_t R, int32_t V) {
  if (!verify_sizes_ok(B, R, V)) return 0;
  return accept_layout(B, R, V).total;
}

ds_status ds_verify_greedy(const float* logits, int32_t B, int32_t R, int32_t V,
                           const int32_t* draft, int32_t* out, int32_t* n_out,
                           void* workspace, size_t ws_bytes, ds_stream_t stream) {
  if (!verify_sizes_ok(B, R, V)) return DS_ERR_INVALID_ARG;
  AcceptProblem pr{logits, B, R, V, true, 1.0, nullptr, draft, nullptr, nullptr, out, n_out};
  return verify_call(pr, workspace, ws_bytes, stream);
}

ds_status ds_verify_sample(const float* logits, int32_t B, int32_t R, int32_t V,
                           double T, const double* qd, const int32_t* draft,
                           const double* u_acc, const double* u_res, int32_t* out,
                           int32_t* n_out, void* workspace, size_t ws_bytes,
                           ds_stream_t stream) {
  if (!verify_sizes_ok(B, R, V)) return DS_ERR_INVALID_ARG;
  if (!(T > 0.0) || !(T < HUGE_VAL)) return DS_ERR_INVALID_ARG;   // finite and positive
  if (!u_res || (R > 1 && (!qd || !u_acc))) return DS_ERR_INVALID_ARG;
  AcceptProblem pr{logits, B, R, V, false, T, qd, draft, u_acc, u_res, out, n_out};
  return verify_call(pr, workspace, ws_bytes, stream);
}

ds_status ds_workspace_status(const void* workspace, ds_stream_t stream) {
  if (!workspace || !aligned(workspace, 256)) return DS_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DS_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return DS_ERR_CUDA;
  if (word & kStatusTimeout) return DS_ERR_TIMEOUT;
  if (word & kStatusCheck) return DS_ERR_DEVICE_CHECK;
  return DS_OK;
}

const char* ds_status_string(ds_status s) {
  switch (s) {
    case DS_OK: return "DS_OK";
    case DS_ERR_INVALID_ARG: return "DS_ERR_INVALID_ARG";
    case DS_ERR_UNSUPPORTED: return "DS_ERR_UNSUPPORTED";
    case DS_ERR_WORKSPACE: return "DS_ERR_WORKSPACE";
    case DS_ERR_CUDA: return "DS_ERR_CUDA";
    case DS_ERR_TIMEOUT: return "DS_ERR_TIMEOUT";
    case DS_ERR_DEVICE_CHECK: return "DS_ERR_DEVICE_CHECK";
  }
  return "DS_ERR_UNKNOWN";
}

const char* ds_version(void) { return "dsmoe 0.1 sm_103a"; }

}  // extern "C"
