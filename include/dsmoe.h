/*
 * dsmoe.h — C ABI of libdsmoe.so: the decode-step hot path of a speculative-verify
 * Q4 Mixture-of-Experts layer and of the compressed-attention block selection beside it,
 * for one GB300 (sm_103a).
 *
 * Sources (the pages about a DeepSeek V4.1 Flash Q4 fork with a native multi-token drafter):
 *   - "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)", paragraph
 *     "Decode": the 384-expert router as one dispatch, the shared expert's gate+up+SwiGLU
 *     as one kernel, BF16 rounding done inside the producing kernels.
 *   - same page, paragraph "DSpark": with the drafter on, a decode step is a 6-row verify,
 *     and the 6 verify rows share one weight stream.
 *   - same page, paragraph "Decode at depth": compressed attention picks 512 blocks per
 *     layer; layers score only the blocks their mask admits, compact the admitted index
 *     once per row, and take the top 512 with a bounded radix select.
 *   The sizes, the Q4 block format, the score formula and the tie-break are the
 *   workload definitions this library is built against (stated beside each call).
 *
 * Conventions shared by every call:
 *   - Every pointer argument is DEVICE memory owned by the caller (for instance the
 *     storage of a torch tensor), except the argument structs themselves, which live on
 *     the host and are only read during the call. The library allocates nothing; its
 *     only state is the header of the caller's workspace, and, for
 *     ds_moe_verify_forward_noalloc alone, one scratch array per device.
 *   - Calls are asynchronous on `stream` and never synchronise the host, except
 *     ds_workspace_status(), which does.
 *   - Arguments are validated on the host before anything is enqueued. A failed check
 *     returns its ds_status and enqueues nothing. A failed launch returns DS_ERR_CUDA.
 *     No C++ exception crosses this boundary.
 *   - Calls are re-entrant provided concurrent calls use distinct workspaces.
 *   - bf16 and fp16 values are passed as their raw 16-bit patterns (uint16_t).
 */
#ifndef DSMOE_H
#define DSMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that C callers need no CUDA header.
 * NULL means the legacy default stream. */
typedef struct CUstream_st* ds_stream_t;
/* Same object as cudaEvent_t. */
typedef struct CUevent_st* ds_event_t;

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, bad alignment          */
  DS_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement             */
  DS_ERR_WORKSPACE = 3,     /* workspace null, misaligned or smaller than required     */
  DS_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed             */
  DS_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up (reported by status) */
  DS_ERR_DEVICE_CHECK = 6   /* a device-side consistency check failed (by status)      */
} ds_status;

/* ------------------------------------------------------------------------------------
 * Q4 weight matrix (the pages' "Q4 weights"; format as defined for this workload):
 * a logical [rows][K] matrix in blocks of 32 consecutive values along K. Each value is
 * an int4 q in [-8, 7]; each block has one fp16 scale; the dequantised value is
 * scale * q (no offset, no minimum).
 *
 * Planar form (the interchange format, input of ds_q4_tile):
 *   qs : uint8 [rows][K/2]. Block b of a row occupies bytes 16b .. 16b+15. Byte j of a
 *        block holds value 2j in its low nibble and value 2j+1 in its high nibble, each
 *        stored as q + 8 (0..15).
 *   sc : fp16 bits [rows][K/32].
 *
 * Tile-major form (what the MoE kernels stream; written once, at load time, by
 * ds_q4_tile): the same values and scales, 0.5625 bytes per weight as above, in tiles of
 * 16 rows x 64 values (two blocks) of 576 bytes. Tile (t, u) covers rows 16t .. 16t+15
 * and values 64u .. 64u+63. Inside a tile, bytes 16L .. 16L+15 (L = 0..31, g = L / 4,
 * w = L % 4) hold the 4-byte word w (values 8w .. 8w+7 of a block, planar byte order) of:
 * row g of block 0, row g+8 of block 0, row g of block 1, row g+8 of block 1; bytes
 * 512 + 8g .. 512 + 8g+7 hold the fp16 scales of row g / block 0, row g+8 / block 0,
 * row g / block 1, row g+8 / block 1. Tile rows are ordered in groups of G consecutive tile
 * rows (the last group of a matrix may be shorter, n rows); inside a group, by K tile
 * first, then by tile row: tile (t, u) of a matrix with T = K/64 sits at tile index
 *   (t - t % G) * T + u * n + t % G,   n = min(G, rows/16 - (t - t % G)),
 * i.e. byte 576 * that index. G = 1 gives plain row-major tiles. The MoE layer's gate and
 * up matrices use G = 1, its down matrices G = DS_Q4_DOWN_GROUP.
 * For a stack of E experts both forms are [E][rows][...], expert-major; each expert's
 * matrix is tiled on its own.
 * ---------------------------------------------------------------------------------- */
typedef struct {
  const uint8_t* qs;
  const uint16_t* sc;
} ds_q4;

/* A Q4 matrix (or expert stack) in the tile-major form; 16-byte aligned. */
typedef struct {
  const void* tiles;
} ds_q4_tiled;

/* Bytes of the tile-major form of a [rows][K] Q4 matrix (rows * K * 9 / 16), or 0 when
 * rows is not a positive multiple of 16 or K not a positive multiple of 64. */
size_t ds_q4_tiled_bytes(int64_t rows, int32_t K);

/* Tile rows per group of the down-projection matrices in the tile-major form. */
#define DS_Q4_DOWN_GROUP 16

/* Writes the tile-major form, with groups of `group` tile rows (1 ..  65536), of n_mats
 * planar matrices [rows][K] stored one after another in `src` (an expert stack:
 * n_mats = E) to `dst` (device memory, >= ds_q4_tiled_bytes(n_mats * rows, K), 16-byte
 * aligned), asynchronously on `stream`. A pure rearrangement of bytes: every nibble and
 * every scale is copied unchanged. src.qs must be 4-byte aligned and src.sc 2-byte
 * aligned. Errors: DS_ERR_INVALID_ARG (null or misaligned pointer, sizes, group),
 * DS_ERR_WORKSPACE (dst_bytes too small), DS_ERR_CUDA. */
ds_status ds_q4_tile(const ds_q4* src, int32_t n_mats, int64_t rows, int32_t K, int32_t group,
                     void* dst, size_t dst_bytes, ds_stream_t stream);

/* One MoE layer: E routed experts + 1 shared expert, each with gate and up [I][H] (tile-
 * major, groups of 1) and down [H][I] (tile-major, groups of DS_Q4_DOWN_GROUP), and a bf16
 * router [E][H].
 * Limits: H and I multiples of 32, 64 <= H <= 16384, 64 <= I <= 8192, 1 <= top_k <= 16,
 * top_k <= E <= 1024 (else DS_ERR_INVALID_ARG). This build's kernels also need H and I
 * to be multiples of 64 (else DS_ERR_UNSUPPORTED). */
typedef struct {
  int32_t hidden;      /* H                                                   */
  int32_t n_experts;   /* E (routed)                                          */
  int32_t inter;       /* I (expert intermediate size)                        */
  int32_t top_k;       /* k                                                   */
  const uint16_t* router_w;              /* bf16 [E][H]                       */
  ds_q4_tiled gate, up, down;            /* routed: gate, up [E][I][H]; down [E][H][I] */
  ds_q4_tiled sh_gate, sh_up, sh_down;   /* shared: gate, up [I][H]; down [H][I]      */
} ds_moe_layer;

/* Bytes of workspace ds_moe_verify_forward needs for this layer and R rows, or 0 when
 * the call would refuse the layer's sizes or R (DS_ERR_INVALID_ARG or
 * DS_ERR_UNSUPPORTED). Host-only: pointers and the device's shared-memory capacity are
 * not examined. The workspace must be 256-byte aligned. */
size_t ds_moe_workspace_size(const ds_moe_layer* layer, int32_t R);

/* One speculative-verify step of one MoE layer for R = 1..6 rows (the pages' 6-row
 * verify, paragraph "DSpark"). For every row r:
 *   z_e = sum_i x[r][i] * router_w[e][i]  (fp32 accumulation), s_e = sigmoid(z_e);
 *   the k experts with the largest s_e (ties to the lower index) in rank order, with
 *   weights w_j = s_j / sum of the k selected s;
 *   for the shared expert and each selected expert e:
 *     h = bf16_rne( silu(Wg_e x_r) * (Wu_e x_r) ),   o = Wd_e h   (fp32 accumulation);
 *   y[r] = bf16_rne( o_shared + sum_j w_j * o_j ), summed in rank order.
 * Every Q4 weight byte of the shared expert and of the union of the experts selected by
 * the R rows is read from HBM once per call and applied to every row that uses it.
 * A row's results do not depend on R or on the other rows: an R-row call writes the same
 * bytes as R one-row calls.
 *   x        : bf16 [R][H]                        (input)
 *   y        : bf16 [R][H]                        (output)
 *   topk_idx : int32 [R][k], expert ids in rank order (output)
 *   topk_w   : fp32 [R][k], renormalised weights  (output)
 *   workspace: >= ds_moe_workspace_size bytes, 256-byte aligned; its contents on entry
 *              are ignored and it must not be used by another call in flight.
 * Errors: DS_ERR_INVALID_ARG (null pointer, R outside 1..6, sizes outside the limits,
 * tiles not 16-byte aligned, misaligned x/y), DS_ERR_WORKSPACE, DS_ERR_UNSUPPORTED (H or
 * I not a multiple of 64, or the device's shared memory too small for the kernel's
 * stages), DS_ERR_CUDA. */
ds_status ds_moe_verify_forward(const ds_moe_layer* layer, const uint16_t* x, int32_t R,
                                uint16_t* y, int32_t* topk_idx, float* topk_w,
                                void* workspace, size_t ws_bytes, ds_stream_t stream);

/* Same as ds_moe_verify_forward, and in addition records caller-created events on
 * `stream` right after each kernel of the call, for per-kernel timing:
 *   marks[0] after the prologue that zeroes the workspace header; marks[1] and marks[2]
 *   after the layer's kernel (router, gate+up+SwiGLU, down projection and combine run as
 *   one kernel, so there is nothing to record between them).
 * `marks` may be NULL and any entry may be NULL (skipped). The events must belong to the
 * stream's device. Errors as ds_moe_verify_forward; DS_ERR_CUDA if recording fails. */
ds_status ds_moe_verify_forward_marked(const ds_moe_layer* layer, const uint16_t* x,
                                       int32_t R, uint16_t* y, int32_t* topk_idx,
                                       float* topk_w, void* workspace, size_t ws_bytes,
                                       ds_stream_t stream, const ds_event_t marks[3]);

/* Byte offset, inside a workspace sized by ds_moe_workspace_size(layer, R), of the bf16
 * array h [R][1 + k][I] that ds_moe_verify_forward leaves there (slot 0 = shared expert,
 * slot j + 1 = the row's rank-j expert): the rounded SwiGLU activations, kept for
 * inspection. Within each group of 8 consecutive values the order is the tensor-core
 * operand order v0, v4, v1, v5, v2, v6, v3, v7. Valid once the call has completed on its
 * stream and until the workspace is reused. Returns (size_t)-1 when the layer or R is
 * invalid. */
size_t ds_moe_workspace_h_offset(const ds_moe_layer* layer, int32_t R);

/* Bytes of the scratch array that ds_moe_verify_forward_noalloc uses, one per device,
 * reserved with the library's kernels (4 MiB: the verify layer of hidden 4096, 384
 * experts, intermediate 1024, top-8 needs 1.0 MiB at R = 6). */
#define DS_NOALLOC_SCRATCH_BYTES (4u << 20)

/* ds_moe_verify_forward without a workspace argument, for callers that cannot allocate
 * device memory at call time: a plain C host loop that embeds one layer and owns no
 * device allocator, or a server whose device memory is fully committed to a pre-reserved
 * pool, where a cudaMalloc would fail or synchronise the device in mid-step. The paper
 * has no counterpart to this call; it computes exactly what ds_moe_verify_forward
 * computes, with the same kernels, and differs only in where its scratch lives.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library routine): it
 * runs on a __device__ array of DS_NOALLOC_SCRATCH_BYTES inside the library, one per
 * device. The first call with a given device current resolves that array's address
 * (and, under lazy module loading, loads the library's kernels); make that first call
 * before any stream capture. All calls on a device share the one array: calls whose work
 * overlaps on the GPU (two streams, two host threads) race on it and give wrong results;
 * serialise them on one stream. The call clears, on `stream`, every part of the array
 * that must start at zero, so a previous call's leftovers do not matter.
 * Arguments, layouts and results as ds_moe_verify_forward; every output buffer is the
 * caller's. Errors: DS_ERR_WORKSPACE, decided on the host before any CUDA call, when
 * ds_moe_workspace_size(layer, R) > DS_NOALLOC_SCRATCH_BYTES; when that size is 0, the
 * status ds_moe_verify_forward gives the layer (DS_ERR_INVALID_ARG or
 * DS_ERR_UNSUPPORTED); DS_ERR_CUDA when the array's address cannot be resolved; otherwise those of ds_moe_verify_forward. The device-side outcomes
 * (DS_ERR_TIMEOUT, DS_ERR_DEVICE_CHECK) are read with ds_noalloc_status().
 * The array's address is resolved once per device and kept for the life of the process;
 * a cudaDeviceReset() invalidates it, so the call must not be used after a reset. */
ds_status ds_moe_verify_forward_noalloc(const ds_moe_layer* layer, const uint16_t* x,
                                        int32_t R, uint16_t* y, int32_t* topk_idx,
                                        float* topk_w, ds_stream_t stream);

/* Synchronises `stream`, then reads the status word that the kernels of the last
 * ds_moe_verify_forward_noalloc call on the current device left at the start of its
 * scratch array: DS_OK, DS_ERR_TIMEOUT or DS_ERR_DEVICE_CHECK, as ds_workspace_status()
 * reports them for a caller workspace. DS_ERR_CUDA when the synchronise, the copy or the
 * address lookup fails. Allocates nothing. */
ds_status ds_noalloc_status(ds_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Block selection for compressed sparse attention (the pages' paragraph "Decode at
 * depth"), batched over L layers and R query rows. For layer l and row r, block b is
 * admitted when b < limit[l][r] and bit (b % 32) of mask[l][r][b / 32] is set. For every
 * admitted block the score is
 *   d_h = fmaf chain over i = 0..D-1 ascending of q[l][r][h][i] * key[l][b][i], from 0.0f;
 *   s   = fmaf chain over h = 0..Hh-1 ascending of head_w[l][r][h] * max(d_h, +0.0f),
 *         from +0.0f;
 * (bf16 inputs widened exactly to fp32; every step one correctly rounded fp32 fma).
 * The selection is the top_k admitted blocks by (s descending, b ascending), with -0.0
 * equal to +0.0, written in ascending b; when fewer than top_k blocks are admitted, all
 * of them are selected and the rest of the row is -1.
 * Limits: 1 <= L, 1 <= R <= 8, 1 <= Hh <= 16, D == 128, 1 <= N <= 2^24,
 * 1 <= top_k <= 2048, 0 <= limit <= N. NaN inputs are a caller error (not checked).
 * ---------------------------------------------------------------------------------- */
typedef struct {
  int32_t n_layers;      /* L                     */
  int32_t n_rows;        /* R                     */
  int32_t n_heads;       /* Hh                    */
  int32_t head_dim;      /* D (must be 128)       */
  int32_t n_blocks;      /* N                     */
  int32_t top_k;         /* 512 in the workload   */
  const uint16_t* keys;  /* bf16 [L][N][D], layer l at keys + l * key_layer_stride elements */
  int64_t key_layer_stride; /* elements between layers, >= N * D, multiple of 8            */
  const uint16_t* q;     /* bf16 [L][R][Hh][D]     */
  const float* head_w;   /* fp32 [L][R][Hh]        */
  const uint32_t* mask;  /* uint32 [L][R][ceil(N/32)] */
  const int32_t* limit;  /* int32 [L][R]           */
  int32_t flags;         /* 0, or DS_SELECT_CANONICAL_SCORES | DS_SELECT_KEEP_WORKSPACE */
} ds_select_args;

/* ds_select_args.flags: compute every admitted block's score in the canonical order on
 * CUDA cores instead of the default tensor-core scoring with exact re-scoring of the
 * candidates near the threshold. Both give the same selection; the default is faster. */
#define DS_SELECT_CANONICAL_SCORES 1
/* ds_select_args.flags: leave the scores, key norms and union lists in the workspace for
 * inspection (below). Without it the top-k drops them from L2 once it has read them (no
 * write-back to memory), and their workspace bytes are undefined after the call. */
#define DS_SELECT_KEEP_WORKSPACE 2

/* Bytes of workspace ds_select_blocks needs, or 0 when the arguments are invalid. */
size_t ds_select_workspace_size(const ds_select_args* args);

/* Runs scoring of admitted blocks, compaction of the admitted index once per row and the
 * bounded radix top-k for all L x R (layer, row) pairs in one call.
 *   sel    : int32 [L][R][top_k], selected blocks ascending, -1 padded (output)
 *   nsel   : int32 [L][R], min(top_k, admitted count)                  (output)
 *   cidx   : int32 [L][R][N], admitted blocks ascending (output; may be NULL)
 *   ccount : int32 [L][R], admitted count                (output; may be NULL)
 * cidx and ccount must be both NULL or both non-NULL.
 * Errors: DS_ERR_INVALID_ARG (null pointer, sizes outside the limits, keys not 16-byte
 * aligned), DS_ERR_WORKSPACE, DS_ERR_CUDA. */
ds_status ds_select_blocks(const ds_select_args* args, int32_t* sel, int32_t* nsel,
                           int32_t* cidx, int32_t* ccount, void* workspace,
                           size_t ws_bytes, ds_stream_t stream);

/* Same as ds_select_blocks, and in addition records caller-created events on `stream`
 * right after each kernel: marks[0] after compaction, marks[1] after scoring, marks[2]
 * after the top-k select. NULL array or entries are skipped. */
ds_status ds_select_blocks_marked(const ds_select_args* args, int32_t* sel, int32_t* nsel,
                                  int32_t* cidx, int32_t* ccount, void* workspace,
                                  size_t ws_bytes, ds_stream_t stream,
                                  const ds_event_t marks[3]);

/* Parts of a select workspace that a completed tensor-core-mode call with
 * DS_SELECT_KEEP_WORKSPACE leaves for inspection, at the byte offsets
 * ds_select_workspace_offset returns (NS = N rounded up to a multiple of 32):
 *   DS_SELECT_WS_UNION       int32 [L][N]: per layer, the blocks some row admits, ascending
 *                            (the first count entries are valid);
 *   DS_SELECT_WS_UNION_COUNT int32 [L]: that count;
 *   DS_SELECT_WS_SCORES      fp32 [L][R][NS]: the tensor-core score s of union entry e for
 *                            row r (-inf where the row does not admit it). A row whose
 *                            candidates overflow the bounded re-score holds canonical
 *                            scores here instead;
 *   DS_SELECT_WS_KEY_NORMS   fp32 [L][NS]: an upper bound kn of the union entry's key norm;
 *   DS_SELECT_WS_ROW_SCALES  fp32 [L][R]: G, an upper bound of 2^-13 * sum_h |w_h| ||q_h||.
 * The selection treats the canonical score as lying within kn * G of s (rounded outward).
 * Valid once the call has completed and until the workspace is reused. */
#define DS_SELECT_WS_UNION 0
#define DS_SELECT_WS_UNION_COUNT 1
#define DS_SELECT_WS_SCORES 2
#define DS_SELECT_WS_KEY_NORMS 3
#define DS_SELECT_WS_ROW_SCALES 4

/* Byte offset of workspace part `part` for a call with these arguments that passes
 * (with_compacted != 0) or does not pass its own cidx / ccount; (size_t)-1 when the
 * arguments or the part are invalid. Host-only. */
size_t ds_select_workspace_offset(const ds_select_args* args, int32_t with_compacted,
                                  int32_t part);

/* ------------------------------------------------------------------------------------
 * Sparse attention over the selected blocks (page "DeepSeek V4.1F Q4 on M3 Ultra with
 * native DSpark MTP (40tps / 800tps)", paragraph "Decode at depth": each layer attends to
 * the 512 blocks its selection picks). The pages stop at the selection; the arithmetic is
 * the plain reading: for layer l, row r and query head h,
 *   s_t = q_{l,r,h} . k_{l,t} / sqrt(D) over the tokens t of the row's selected blocks
 *         (tokens block_tokens * b .. block_tokens * b + block_tokens - 1 of block b),
 *   p = softmax(s),  out_{l,r,h} = bf16_RNE(sum_t p_t v_{l,t}),
 * all heads of a row sharing each token's key and value; a row with no selected block
 * gets 0. Sums in fp32 on the tensor cores (bf16 products exact; p carried as a bf16 high
 * and low part), so the result is not bit-exact with an fp64 evaluation. */
typedef struct {
  int32_t n_layers;       /* L                                                       */
  int32_t n_rows;         /* R, 1 .. 8                                               */
  int32_t n_heads;        /* Hq query heads, 1 .. 16                                 */
  int32_t head_dim;       /* D, 128                                                  */
  int32_t n_blocks;       /* N blocks per layer                                      */
  int32_t block_tokens;   /* tokens per block: 1, 2, 4, 8 or 16                      */
  int32_t top_k;          /* entries of sel per row, 1 .. 2048                       */
  const uint16_t* q;      /* bf16 [L][R][Hq][D]                                      */
  const uint16_t* k;      /* bf16 [L][N * block_tokens][D], layer stride below        */
  const uint16_t* v;      /* same layout as k                                        */
  int64_t kv_layer_stride;   /* values between layers of k and v (>= N*block_tokens*D) */
  const int32_t* sel;     /* int32 [L][R][top_k]: block ids (as written by
                             ds_select_blocks), -1 for none; ids >= N are skipped     */
} ds_attn_args;

/* Workspace bytes for these arguments (0 when they are invalid). Host-only. */
size_t ds_attn_workspace_size(const ds_attn_args* args);
/* out: bf16 [L][R][Hq][D] (device, 16-byte aligned); q, k, v 16-byte aligned; workspace
 * 256-byte aligned of ds_attn_workspace_size bytes. DS_ERR_INVALID_ARG outside the limits
 * above, DS_ERR_UNSUPPORTED for head_dim != 128. */
ds_status ds_sparse_attention(const ds_attn_args* args, uint16_t* out, void* workspace,
                              size_t ws_bytes, ds_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Paired Q8 projections (page "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP
 * (40tps / 800tps)", paragraph "DSpark": the 6 verify rows share one weight stream
 * through paired Q8 projections). Format as defined for this workload: a logical
 * [rows][K] matrix in blocks of 32 consecutive int8 values (two's complement) along K,
 * one fp16 scale per block, value = scale * q.
 *   Planar interchange form: qs int8 [rows][K], sc fp16 bits [rows][K/32].
 *   Tile-major form (what ds_q8_project streams; written by ds_q8_tile): tiles of 16 rows
 *   x 64 values, 1088 bytes each, ordered by 16-row unit, then K tile. Within a tile,
 *   block j (0, 1) occupies bytes 512 j .. 512 j + 511: lane L = 4g + q (g, q < 8, 4) holds
 *   at 512 j + 16 L the int8 values k = 4q .. 4q+3 of rows g and g + 8 of the block's first
 *   16 values, then the same of its last 16 values (4 bytes each, k ascending). Bytes
 *   1024 + 8 g hold the fp16 scales (row g block 0, row g+8 block 0, row g block 1,
 *   row g+8 block 1). A pure rearrangement (1.0625 bytes per weight in both forms). */
typedef struct {
  const int8_t* qs;
  const uint16_t* sc;
} ds_q8;
typedef struct {
  const void* tiles;   /* 16-byte aligned */
} ds_q8_tiled;

/* Bytes of the tile-major form of a [rows][K] Q8 matrix (0 when rows is not a positive
 * multiple of 16 or K not a positive multiple of 64). */
size_t ds_q8_tiled_bytes(int64_t rows, int32_t K);
/* Planar -> tile-major on the device (qs, sc and dst 16-byte aligned device memory,
 * dst_bytes >= ds_q8_tiled_bytes). DS_ERR_INVALID_ARG for nulls, misalignment, or sizes
 * outside rows % 16 == 0, K % 64 == 0, rows <= 2^24, K <= 65536; DS_ERR_WORKSPACE when dst is
 * too small. */
ds_status ds_q8_tile(const ds_q8* src, int64_t rows, int32_t K, void* dst, size_t dst_bytes,
                     ds_stream_t stream);
/* Workspace of ds_q8_project: the 256-byte status header. */
size_t ds_q8_workspace_size(void);
/* y[r][i] = bf16_RNE(sum_k W[i][k] * x[r][k]) for r < R: x bf16 [R][K], y bf16 [R][rows]
 * (device, 16-byte aligned), 1 <= R <= 8. Every weight byte is read from HBM once for all
 * R rows; products are exact and summed in fp32 in an order that does not depend on R,
 * so an R-row call writes the same bytes as R one-row calls. DS_ERR_INVALID_ARG outside
 * the format (rows % 16, K % 32, ranges as for ds_q8_tile, R); DS_ERR_UNSUPPORTED for a
 * valid K this kernel does not run (K not a multiple of 1024, or R x K activations beyond
 * its shared memory: R x K x 2 bytes must leave room for its ring). */
ds_status ds_q8_project(const ds_q8_tiled* w, int64_t rows, int32_t K, const uint16_t* x,
                        int32_t R, uint16_t* y, void* workspace, size_t ws_bytes,
                        ds_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Verify acceptance (page "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP
 * (40tps / 800tps)", paragraph "DSpark": a decode step verifies the last committed token
 * and R - 1 drafts in one pass; greedy decode gives the same output as without the
 * drafter, and at temperature > 0 the step does exact speculative sampling).
 *
 * B independent steps of R rows (1 <= R <= 16) over a vocabulary of V tokens
 * (1 <= V <= 2^24), 1 <= B <= 4096. Row r's logits predict the token after row r's
 * input, so draft r (r < R - 1) is checked against row r.
 *   logits  fp32 [B][R][V], finite.
 *   draft   int32 [B][R-1], tokens in [0, V) (NULL when R == 1). A draft outside the
 *           vocabulary is rejected and reported as DS_ERR_DEVICE_CHECK by
 *           ds_workspace_status.
 *   out     int32 [B][R]: the emitted tokens of each step (the kept drafts, then the one
 *           token the target adds), -1 after them.
 *   n_out   int32 [B]: how many tokens each step emitted (1 .. R).
 * Greedy: every row's argmax, ties to the lowest token id; drafts are kept while they
 * equal their row's argmax; the first mismatching row, or the last row, adds its argmax.
 * Sampling at temperature T (finite, > 0; else DS_ERR_INVALID_ARG), every decision in
 * fp64: p_r = softmax(logits_r / T); draft d of row r is kept iff u_acc * qd_r[d] < p_r[d];
 * at the first rejection the added token is drawn from max(p_r - qd_r, 0) (from p_r if
 * that is zero everywhere), after R - 1 kept drafts from p_{R-1}; a draw with u takes the
 * smallest token whose cumulative weight (token order) exceeds u times the total weight,
 * else the last token with a positive weight.
 *   qd      fp64 [B][R-1][V]: the drafter's proposal distributions (NULL when R == 1).
 *   u_acc   fp64 [B][R-1] in [0, 1): the acceptance uniforms (NULL when R == 1).
 *   u_res   fp64 [B][R] in [0, 1): the uniforms of the added token (only the one of the
 *           row it is drawn from is read).
 * Sums over the vocabulary are taken in a fixed parallel order, so a draw whose target
 * lies within rounding (about 1e-15 of the total) of a cumulative boundary may differ
 * from a sequential fp64 evaluation.
 * The workspace (ds_verify_workspace_size, 256-byte aligned) holds per-chunk partials
 * and the status word. */
size_t ds_verify_workspace_size(int32_t B, int32_t R, int32_t V);
ds_status ds_verify_greedy(const float* logits, int32_t B, int32_t R, int32_t V,
                           const int32_t* draft, int32_t* out, int32_t* n_out, void* workspace,
                           size_t ws_bytes, ds_stream_t stream);
ds_status ds_verify_sample(const float* logits, int32_t B, int32_t R, int32_t V, double T,
                           const double* qd, const int32_t* draft, const double* u_acc,
                           const double* u_res, int32_t* out, int32_t* n_out, void* workspace,
                           size_t ws_bytes, ds_stream_t stream);

/* Synchronises `stream`, then reads the status word that the kernels of the last call on
 * this workspace left in its header: DS_OK, DS_ERR_TIMEOUT (a bounded device wait gave
 * up) or DS_ERR_DEVICE_CHECK (a device consistency check failed, e.g. an index out of
 * range; the offending access was skipped). DS_ERR_CUDA when the synchronise fails.
 * The word is reset at the start of every call that uses the workspace. */
ds_status ds_workspace_status(const void* workspace, ds_stream_t stream);

/* Static, NUL-terminated name of a status code. */
const char* ds_status_string(ds_status s);

/* Library version string, e.g. "dsmoe 0.1 sm_103a". */
const char* ds_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSMOE_H */
