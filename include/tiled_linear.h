/*
 * tiled_linear.h -- C ABI of a host-streamed, output-tiled linear operator for
 * one GB300 GPU (sm_103a).
 *
 * The operator is Y = X.W with W [K, M] too large to keep on the device.  W is
 * split along its output dimension into N tiles W_1..W_N of Mi = M/N columns;
 * the forward pass computes Y_i = X.W_i one tile at a time and the column
 * blocks Y_i together are Y, with no cross-tile term (pwwt.cn/news/5430303,
 * "关键技术一: Memory-centric tiling", 核心思想; aicassindra
 * tm_zero_infinity, "Memory-centric tiling: operators bigger than the
 * device").  Each tile lives in pinned host memory and is copied into a ring
 * of device slots up to d tiles ahead of the tile being computed, with the
 * depth rule d >= t_fetch / t_layer (tm_zero_infinity, "Prefetch depth: how
 * far ahead the pipeline must run").  A slot is reused as soon as its last
 * reader finishes (the gathered weights are released after use:
 * gpu_zero_sharding, "End-to-end flow").  Backward fetches every tile again,
 * computes dW_i = X^T.dY_i and writes it back to pinned host memory on a
 * second copy stream while later tiles compute (pwwt.cn/news/5430303,
 * "关键技术三", 后向传播中的重叠), and accumulates dX += dY_i.W_i^T in fp32.
 *
 * Conventions for every function:
 *  - All matrices are row-major, bf16 stored as 16-bit patterns unless stated.
 *  - "_dev" pointers are device memory of the handle's device; "_host"
 *    pointers are pinned host memory (cudaHostAlloc / cudaHostRegister or
 *    tiled_linear_host_alloc).  The caller owns every buffer it passes.
 *  - A `stream` argument is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  Work is enqueued and the call returns; results are
 *    valid once `stream` has completed.
 *  - Errors are returned as tl_status; nothing is thrown across the ABI.  A
 *    CUDA failure inside a call makes the handle sticky-failed: later calls
 *    return TL_ERR_STATE and tiled_linear_last_error() keeps the message.
 *  - A handle is not thread-safe: use one handle per thread.
 *  - No function here allocates device memory; the caller supplies it.
 */
#ifndef TILED_LINEAR_H
#define TILED_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tl_handle tl_handle;

typedef enum {
    TL_OK = 0,
    TL_ERR_INVALID = 1,     /* bad shape, depth, pointer or alignment        */
    TL_ERR_NOT_PINNED = 2,  /* w_host / dw_host is not pinned host memory    */
    TL_ERR_WORKSPACE = 3,   /* workspace too small or misaligned             */
    TL_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed           */
    TL_ERR_TIMEOUT = 5,     /* a kernel's bounded wait gave up (see below)   */
    TL_ERR_STATE = 6,       /* handle already failed, or NULL                */
    TL_ERR_IO = 7           /* a file of the file tier failed (open, read,   */
                            /* write), see tiled_linear_create_file          */
} tl_status;

/* Host storage of W (read) and dW (written).
 *  ROW_MAJOR : logical [K, M] row-major; tile i is a strided column block
 *              (copied with pitched 2-D copies).
 *  TILE_MAJOR: [N][K][Mi]; tile i is one contiguous K*Mi block (copied with
 *              1-D copies, which keep the full host-link bandwidth). */
typedef enum { TL_LAYOUT_ROW_MAJOR = 0, TL_LAYOUT_TILE_MAJOR = 1 } tl_layout;

/* Timings from CUDA events the library records on the streams that run the
 * work, in milliseconds.  The first block describes the LAST forward and
 * backward call: *_gemm_ms are sums of the kernels' own spans on the compute
 * stream, *_h2d_ms / *_d2h_ms sums of the copy spans on the copy streams,
 * *_total_ms the whole call on `stream`.  The sum_* block adds the same
 * quantities over every timed call since the handle was created or
 * tiled_linear_reset_stats was called: fwd_timed_calls / bwd_timed_calls of
 * the fwd_calls / bwd_calls made.  Every call is timed unless
 * tiled_linear_set_timing says otherwise; the first block then describes
 * the last timed call.  Each call launches one GEMM per tile (and, in the
 * backward, one dX GEMM per tile group); bwd_gemm_ms = bwd_dw_gemm_ms +
 * bwd_dx_gemm_ms. */
typedef struct {
    int32_t n_tiles;
    int32_t depth;            /* d used by the call                           */
    int32_t fwd_valid, bwd_valid;
    float fwd_total_ms, fwd_gemm_ms, fwd_h2d_ms;
    float bwd_total_ms, bwd_dw_gemm_ms, bwd_dx_gemm_ms, bwd_h2d_ms, bwd_d2h_ms;
    float fwd_wait_ms;        /* fwd_total - fwd_gemm: compute stream idle    */
    float bwd_wait_ms;        /* bwd_total - both GEMM sums                   */
    int64_t fwd_h2d_bytes, bwd_h2d_bytes, bwd_d2h_bytes;
    int32_t fwd_launches, bwd_launches;   /* kernels launched by the call     */
    int64_t fwd_calls, bwd_calls;
    double sum_fwd_total_ms, sum_fwd_gemm_ms, sum_fwd_h2d_ms;
    double sum_bwd_total_ms, sum_bwd_dw_gemm_ms, sum_bwd_dx_gemm_ms, sum_bwd_h2d_ms, sum_bwd_d2h_ms;
    double sum_bwd_gemm_ms;
    float bwd_gemm_ms;
    int32_t staging_slots;    /* device dW staging slots of the handle       */
    int32_t bwd_reused_tiles; /* tiles the last backward took from the ring
                                 instead of fetching (tiled_linear_set_tile_reuse) */
    int64_t fwd_timed_calls, bwd_timed_calls; /* calls in the sum_* block */
    int32_t timing_every;     /* see tiled_linear_set_timing */
    float fwd_h2d_max_ms;     /* slowest single tile copy of the last forward */
} tl_stats;

/* Device workspace bytes for (K, M, N, d): (min(d,N-1)+1) weight slots and
 * min(2,N) gradient staging slots of K*(M/N) bf16 each, plus a 4 KiB header
 * (the kernels' error word and tile counter).  d = -1 (automatic depth): the
 * most the handle can use, N weight slots and N staging slots; create accepts
 * any workspace down to 2 weight and min(2,N) staging slots and carves as
 * many slots as fit.  Returns 0 if the arguments are invalid. */
size_t tiled_linear_workspace_bytes(int64_t K, int64_t M, int32_t N, int32_t d);

/* Create a handle on `device`.
 *  K, M, N : W is [K, M] bf16, split into N tiles of Mi = M/N columns.
 *            Requires K >= 8, K % 8 == 0, M % N == 0, Mi % 8 == 0 (16-byte
 *            row pitches for the tensor-memory-access engine).
 *  d       : tiles fetched ahead of the one being computed (ring of d+1
 *            slots; d >= N-1 keeps every tile resident).  d = 0 serialises
 *            copy and compute.  d = -1 (automatic) picks, after the first
 *            forward call, d = ceil(t_fetch / t_layer) with t_layer that
 *            call's mean per-tile GEMM time and t_fetch its slowest tile copy
 *            plus a stall allowance (50 ms by default, see
 *            tiled_linear_set_stall_allowance), bounded by the weight slots
 *            the workspace holds; every staging slot that fits is used.
 *  w_host  : pinned host W (read by every call; must not change while a
 *            call is in flight).  dw_host: pinned host dW (overwritten by
 *            every backward call).  Both in tiled_linear_create's layout:
 *            TL_LAYOUT_ROW_MAJOR.  May alias nothing else the call writes.
 *  workspace_dev, workspace_bytes: device memory, 256-byte aligned, at least
 *            tiled_linear_workspace_bytes(K, M, N, d); owned by the caller,
 *            used until tiled_linear_destroy returns.
 * Each call launches one GEMM per tile (and per GEMM in the backward),
 * ordered against the copy streams by CUDA events.
 * Errors: TL_ERR_INVALID (shapes/pointers), TL_ERR_NOT_PINNED,
 * TL_ERR_WORKSPACE, TL_ERR_CUDA.  On error *out is set to NULL. */
tl_status tiled_linear_create(tl_handle **out, int64_t K, int64_t M, int32_t N, int32_t d,
                              const void *w_host, void *dw_host,
                              void *workspace_dev, size_t workspace_bytes, int device);

/* As tiled_linear_create, with W and dW stored tile-major [N][K][Mi]. */
tl_status tiled_linear_create_tilemajor(tl_handle **out, int64_t K, int64_t M, int32_t N,
                                        int32_t d, const void *w_host, void *dw_host,
                                        void *workspace_dev, size_t workspace_bytes,
                                        int device);

/* File tier: W and dW live in files instead of host memory, one tier further
 * from the GPU (ZeRO-Infinity keeps them on NVMe and moves each tile up one
 * tier at a time: NVMe -> pinned CPU buffers with direct I/O -> GPU, the
 * stages overlapping on different tiles; "Overlap-centric design", and the
 * direct-I/O-into-pinned-buffers rule of memory-centric tiling, "Pitfalls").
 *  w_path  : file holding W tile-major [N][K][Mi] bf16 (N * K*Mi*2 bytes at
 *            least), opened read-only with O_DIRECT.
 *  dw_path : file that receives dW in the same layout, opened with O_DIRECT
 *            (created, and extended to N tiles if shorter).
 *  host_slots (2..64): pinned host slots per direction, each one tile.  Reader
 *            threads read up to host_slots tiles ahead of the host->device
 *            copies (which run up to d tiles ahead of the GEMMs); the
 *            device->host copies of dW land in the other host_slots slots,
 *            which writer threads store to dw_path.
 *  io_threads (1..64): threads per direction; each tile is read / written
 *            as 16 MiB direct-I/O requests spread over them.
 * A tile (K * M/N * 2 bytes) must be a multiple of 4096 bytes.  The other
 * arguments and the workspace are as tiled_linear_create_tilemajor.  The
 * handle takes no host optimizer.  A forward or backward call returns once its last copy is
 * enqueued, so the calling thread waits for the tile reads (the GPU works on
 * the tiles already there meanwhile), and a backward also waits for free dW
 * slots.  dW is in dw_path only after tiled_linear_file_sync.
 * Errors: as tiled_linear_create, and TL_ERR_IO (a file cannot be opened
 * with direct I/O, is too short, or the pinned slots cannot be had).  A read
 * or write that fails later makes the handle fail with TL_ERR_IO. */
tl_status tiled_linear_create_file(tl_handle **out, int64_t K, int64_t M, int32_t N, int32_t d,
                                   const char *w_path, const char *dw_path, int32_t host_slots,
                                   int32_t io_threads, void *workspace_dev, size_t workspace_bytes,
                                   int device);

/* Block until every dW tile of the backward calls made so far is in dw_path.
 * Call it after the calls' stream has been synchronised (it does not wait for
 * work still queued on the device, only for the writers).  TL_ERR_INVALID if
 * the handle has no file tier, TL_ERR_IO if a write failed. */
tl_status tiled_linear_file_sync(tl_handle *h);

/* Counters of the file tier since the handle was created. */
typedef struct {
    int64_t read_bytes, write_bytes;   /* W bytes read, dW bytes written       */
    double read_seconds, write_seconds; /* summed wall time of the tile I/O    */
    double fetch_wait_seconds;         /* calls waiting for a tile to be read  */
    double writeback_wait_seconds;     /* calls waiting for a free dW slot     */
    int32_t host_slots, io_threads;
} tl_file_stats;
tl_status tiled_linear_file_stats(const tl_handle *h, tl_file_stats *out);

/* Forward: y_dev[T, M] (bf16, ld M) = x_dev[T, K] (bf16, ld K) . W, tile by
 * tile, fp32 accumulation, round-to-nearest-even to bf16.  T >= 0 (T = 0 is
 * a no-op).  Weight copies may begin before earlier work on `stream`
 * finishes (they only read w_host).  Errors: TL_ERR_INVALID, TL_ERR_STATE,
 * TL_ERR_CUDA, TL_ERR_TIMEOUT (a previous call's kernel timed out). */
tl_status tiled_linear_forward(tl_handle *h, int64_t T, const void *x_dev, void *y_dev,
                               void *stream);

/* Backward, tiles in descending order i = N-1 .. 0:
 *   dW_i = X^T . dY_i  (fp32 accumulation, bf16 RNE) -> dw_host tile i
 *   dx_dev[T, K] (fp32, ld K) = sum_i dY_i . W_i^T   (overwritten).  Fixed
 *   summation order: when min(d, N-1) >= 2 and Mi % 64 == 0, tiles go in
 *   groups of g = min(max(2, ceil(8192 / Mi)), d, N-1, 4) consecutive tiles,
 *   (N-1 .. N-g), (N-g-1 .. N-2g), ..., the last group holding what is
 *   left; each group is reduced
 *   in one fp32 accumulator over its columns in ascending order, the first
 *   group stores, later groups add.  Otherwise the first tile stores and
 *   later tiles add one at a time.  The order depends on (N, Mi, d) alone,
 *   not on the schedule (host layout, tile reuse, copy timing).
 * dy_dev is [T, M] bf16 (ld M).  T = 0 writes dW = 0.  dW on the host is
 * complete once `stream` has completed.  Errors as tiled_linear_forward. */
tl_status tiled_linear_backward(tl_handle *h, int64_t T, const void *x_dev,
                                const void *dy_dev, float *dx_dev, void *stream);

/* Synchronise the handle's streams, release its streams and events and free
 * the handle.  The caller's buffers are untouched.  Returns the handle's
 * sticky status (TL_OK if it never failed).  NULL is accepted (TL_OK). */
tl_status tiled_linear_destroy(tl_handle *h);

/* Message of the last failure on h ("" if none); a static message for NULL. */
const char *tiled_linear_last_error(const tl_handle *h);

/* Wait for the handle's last forward and backward calls to finish, check the
 * kernels' timeout word, and fill *out (a tl_stats).  Returns TL_ERR_TIMEOUT
 * if a kernel gave up waiting. */
tl_status tiled_linear_get_stats(tl_handle *h, void *tl_stats_out);

/* Timeline of the last timed forward (backward = 0) or backward call: every
 * GEMM launch and every tile copy that call made, with its start and end in
 * milliseconds from the call's start on its `stream`, from the CUDA events the
 * library records on the stream that ran it (the copy engines' view that a
 * system trace would give).
 *  kind: TL_TRACE_FWD_GEMM / _DW_GEMM / _DX_GEMM (a dX launch over a group of
 *        tiles is listed under the group's lowest tile), TL_TRACE_H2D (a W
 *        tile into the ring; tiles a backward reused from the ring have none),
 *        TL_TRACE_D2H (a dW tile out).
 *  tile: the tile's index in the handle's order (a chain's operators follow
 *        each other).
 * Events are listed GEMMs first, in launch order, then copies in fetch order.
 * A copy can start before the call does (a negative start): a weight fetch
 * waits only for its ring slot, not for earlier work on `stream`.
 * Writes min(*count, capacity) events to out and sets *count to the number
 * there are (0 if no call of that direction was timed).  Waits for that call
 * to finish.  Errors: TL_ERR_INVALID (null handle / count, negative
 * capacity, null out with capacity > 0), TL_ERR_CUDA. */
enum { TL_TRACE_FWD_GEMM = 0, TL_TRACE_DW_GEMM = 1, TL_TRACE_DX_GEMM = 2, TL_TRACE_H2D = 3, TL_TRACE_D2H = 4 };
typedef struct {
    int32_t kind;
    int32_t tile;
    float start_ms, end_ms;
} tl_trace_event;
tl_status tiled_linear_get_trace(tl_handle *h, int32_t backward, tl_trace_event *out, int32_t capacity,
                                 int32_t *count);

/* Wait for every recorded call to finish and zero the sum_* counters. */
tl_status tiled_linear_reset_stats(tl_handle *h);

/* Record the per-launch and per-copy timing events of every `every`-th call
 * only (every >= 1; default 1: all calls).  Each event recorded between two
 * kernels widens the gap between them; on the GPT-scale layer, timing every
 * call costs about 0.8 % of the step.  The call counts, and the start / end
 * of every call, are kept either way.  Errors: TL_ERR_INVALID (every < 1),
 * TL_ERR_STATE. */
tl_status tiled_linear_set_timing(tl_handle *h, int32_t every);

/* Tile reuse across calls -- an opt-in extension; the method itself fetches
 * every tile again for the backward (tm_zero_infinity, "The FLOPs-per-byte
 * test": parameters climb the hierarchy twice per step).  The prefetcher
 * follows the operator sequence: it knows which tiles come next
 * (pwwt.cn/news/5430303, 关键技术三 (1) 动态预取器).  With enable != 0, a
 * backward call takes the tiles its descending order starts with from the
 * ring when the calls before it left them there -- after a forward, the last
 * min(d+1, N) tiles -- instead of fetching them again.  tl_stats reports them
 * as bwd_reused_tiles, and bwd_h2d_bytes drops by as many tiles.  Results are
 * bit-identical to refetching as long as the host W buffer is not written
 * between the calls; writing it there is undefined.  Default: off.  Errors:
 * TL_ERR_STATE on a failed handle. */
tl_status tiled_linear_set_tile_reuse(tl_handle *h, int32_t enable);

/* Stall allowance of the automatic depth (d = -1 at creation), in
 * milliseconds: the time added to the slowest tile copy of the first forward
 * call before the depth rule d = ceil(t_fetch / t_layer) is applied
 * (tm_zero_infinity, "Prefetch depth").  The host link of a shared machine
 * stalls now and then for tens of milliseconds; a ring sized from mean copy
 * times stops the GEMMs for the length of such a stall ("Pitfalls": a
 * mistuned prefetch stalls).  Default 50 ms; 0 applies the rule to the
 * slowest copy alone.  Takes effect if set before the first forward call;
 * ignored at a fixed depth.  Errors: TL_ERR_INVALID (ms < 0 or not finite),
 * TL_ERR_STATE. */
tl_status tiled_linear_set_stall_allowance(tl_handle *h, double ms);

/* --- the optimizer step on the host ----------------------------------------
 * The Adam update runs on the CPU, beside the DRAM holding its state: it is
 * elementwise, about 12 FLOPs against ~24 bytes read and written per
 * parameter, so no host link could hide it behind GPU compute
 * (tm_zero_infinity, "Applying the test: which state can live where").  The
 * state is 12 bytes per parameter: fp32 master weight, first and second
 * moment (gpu_zero_sharding, "The architecture: every piece explained").
 * The update is Adam with bias correction and decoupled weight decay, in
 * fp32, one element at a time:
 *     g  = grad (+ the fp32 accumulator, when gradients were accumulated)
 *     m  = beta1 m + (1 - beta1) g
 *     v  = beta2 v + (1 - beta2) g^2
 *     p  = p - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 *            - lr weight_decay p
 *     w  = bf16 round-to-nearest-even of p (the weights the next pass streams)
 * The pages name Adam and its state but write no formula; this is the
 * textbook update.  No part of it runs on the GPU. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int32_t threads;  /* host threads of the optimizer below (<= 0: all) */
} tl_adam_config;

/* One Adam step (t = step >= 1) over n parameters, in the calling thread:
 * master, m, v fp32 (updated), grad_bf16 the gradient (bf16 bits), grad_acc
 * an fp32 gradient added to it (or NULL), w_bf16 receives the new weights.
 * Errors: TL_ERR_INVALID (null pointers, bad config). */
tl_status tiled_linear_adam_update(const tl_adam_config *cfg, int64_t step, int64_t n, float *master,
                                   float *m, float *v, const float *grad_acc, const void *grad_bf16,
                                   void *w_bf16);

/* A host optimizer attached to a handle (per-tile launch mode; single
 * operator or chain).  Per operator l: master[l], m[l], v[l] (and grad_acc[l]
 * if grad_acc is not NULL) are fp32 host arrays of dims K x M elements, in
 * the same layout as that operator's host W (row-major or tile-major); the
 * caller owns them and initialises master (normally to W) and zeroes m, v.
 * After a backward call:
 *   tiled_linear_optimizer_accumulate: grad_acc (+)= that backward's dW (the
 *     first accumulation after a step overwrites);
 *   tiled_linear_optimizer_step: the Adam step with g = dW (+ grad_acc if it
 *     was filled since the last step), writing master, m, v and the bf16 W in
 *     the handle's host W buffer.
 * Both return at once.  A worker thread takes the tiles in the backward's
 * order as each one's dW lands in host memory, so the update overlaps the
 * GPU's backward of the later tiles.  The handle's later calls wait (on the
 * host) before queuing a copy of a tile's W until its update is done, and
 * before writing a tile's dW until the worker has read the previous one:
 * forward / backward may therefore block the calling thread.  Results are
 * bit-identical to calling tiled_linear_adam_update tile by tile after the
 * backward completes.  Host waits give up after 600 s with TL_ERR_TIMEOUT.
 * Errors: TL_ERR_INVALID (arguments, a handle whose W and
 * dW are in files, accumulate without an accumulator), TL_ERR_STATE (no backward since the last optimizer call, or
 * an optimizer already attached), TL_ERR_CUDA, TL_ERR_TIMEOUT. */
typedef struct tl_optimizer tl_optimizer;
tl_status tiled_linear_optimizer_create(tl_optimizer **out, tl_handle *h, const tl_adam_config *cfg,
                                        float *const *master, float *const *m, float *const *v,
                                        float *const *grad_acc);
tl_status tiled_linear_optimizer_accumulate(tl_optimizer *o);
tl_status tiled_linear_optimizer_step(tl_optimizer *o);
/* Block until every submitted accumulation and step is done. */
tl_status tiled_linear_optimizer_wait(tl_optimizer *o);
/* Steps submitted so far, and host seconds spent updating. */
tl_status tiled_linear_optimizer_stats(const tl_optimizer *o, int64_t *steps, double *busy_seconds);
/* Wait for the submitted work, detach from the handle, free.  Destroy the
 * optimizer before its handle (tiled_linear_destroy detaches it too). */
tl_status tiled_linear_optimizer_destroy(tl_optimizer *o);

/* --- chains of operators: one prefetcher across several linear layers -----
 * A chain of L tiled linear operators, run in sequence by one handle:
 * operator l computes Y_l [T, dims[l+1]] = X_l [T, dims[l]] . W_l with W_l
 * split into n_tiles[l] column tiles, X_0 = x and X_l = Y_{l-1} (bf16).  With
 * L = 2 and dims = {K, 4K, K} this is the FFN's up- and down-projection, the
 * two matrices the tiling splits (tm_zero_infinity, "Memory-centric tiling:
 * operators bigger than the device"), with no activation between them.  One
 * ring serves every operator.  Its prefetcher follows the operator sequence
 * (pwwt.cn/news/5430303, 关键技术三 (1) 动态预取器): the next operator's first
 * tiles are fetched while the current one's last tiles compute, in the
 * forward and in the backward.  Each operator obeys tiled_linear_create's
 * shape rules for (dims[l], dims[l+1], n_tiles[l]); the host W_l and dW_l are
 * tile-major [n_tiles[l]][dims[l]][dims[l+1]/n_tiles[l]], pinned.  A chain
 * handle also serves tiled_linear_destroy, _last_error, _get_stats (n_tiles
 * = all operators' tiles), _reset_stats and _set_tile_reuse.  It runs one
 * launch per tile; tiled_linear_forward / _backward refuse it, and the
 * chain calls refuse a single-operator handle (TL_ERR_INVALID).  L = 1 gives the same results as
 * tiled_linear_create_tilemajor. */

/* Workspace bytes for a chain (as tiled_linear_workspace_bytes, with the ring
 * slots sized for the largest tile and d counted over all operators' tiles);
 * 0 if the arguments are invalid. */
size_t tiled_linear_chain_workspace_bytes(int32_t L, const int64_t *dims, const int32_t *n_tiles,
                                          int32_t d);

/* Create a chain handle.  dims has L+1 entries, n_tiles, w_host and dw_host L
 * each; the arrays are read during the call only, the buffers they point to
 * are used until tiled_linear_destroy.  Errors as tiled_linear_create. */
tl_status tiled_linear_chain_create(tl_handle **out, int32_t L, const int64_t *dims,
                                    const int32_t *n_tiles, int32_t d,
                                    const void *const *w_host, void *const *dw_host,
                                    void *workspace_dev, size_t workspace_bytes, int device);

/* Forward through the chain: y_dev[l] (bf16 [T, dims[l+1]], ld dims[l+1])
 * receives operator l's output, each as tiled_linear_forward computes it.
 * Keep y_dev[0..L-2] for the backward.  Errors as tiled_linear_forward. */
tl_status tiled_linear_chain_forward(tl_handle *h, int64_t T, const void *x_dev,
                                     void *const *y_dev, void *stream);

/* Device scratch bytes the chain backward needs: an fp32 buffer and, for the
 * dY between operators, one bf16 buffer (two for L >= 3, so that a middle
 * operator writes the next dY beside the one it reads), each of
 * T x max(dims[1..L-1]) elements (0 for L = 1). */
size_t tiled_linear_chain_scratch_bytes(int64_t T, int32_t L, const int64_t *dims);

/* Backward through the chain, operators in reverse: operator L-1 takes dy_dev
 * (bf16 [T, dims[L]]) as its dY; operator l < L-1 takes the bf16 RNE of the
 * fp32 dX that operator l+1 produced.  Each operator's dW_l goes to its
 * dw_host as tiled_linear_backward writes it, and dx_dev (fp32 [T, dims[0]])
 * receives operator 0's dX.  Operator l sums its dX over the tile groups that
 * tiled_linear_backward uses for n_tiles[l] tiles at depth d.  y_dev[0..L-2] are the forward's outputs (the
 * inputs X_1..X_{L-1}); for L = 1 y_dev may be NULL.  scratch_dev: 256-byte
 * aligned device memory of at least tiled_linear_chain_scratch_bytes(T, L,
 * dims) bytes (may be NULL for L = 1), used until `stream` completes.
 * Errors as tiled_linear_backward, TL_ERR_WORKSPACE for the scratch. */
tl_status tiled_linear_chain_backward(tl_handle *h, int64_t T, const void *x_dev,
                                      const void *const *y_dev, const void *dy_dev,
                                      float *dx_dev, void *scratch_dev, size_t scratch_bytes,
                                      void *stream);

/* --- resident GEMMs: the three kernels on device-resident operands --------
 * The same kernels the engine launches per tile, for callers that already
 * hold a tile on the device.  fp32 accumulation in tensor memory.  err_dev
 * points to two device int32 words, zeroed by the caller before first use:
 * err_dev[0] is set non-zero if a bounded wait gives up (it is only ever
 * OR-ed into, never cleared); err_dev[1] is the counter the CTAs draw output
 * tiles from (dynamic schedule), which every launch that completes without a
 * timeout leaves at zero -- after a timeout, zero both words again.  Calls
 * that may run at the same time (different streams) need separate err
 * buffers.  Requirements: every leading dimension and column offset a
 * multiple of 8 elements, pointers 16-byte aligned, all sizes >= 1.
 * Errors: TL_ERR_INVALID, TL_ERR_CUDA. */

/* y[T, n] (bf16, ld ldy) = x[T, K] (bf16, ld ldx) . w[K, n] (bf16, ld ldw). */
tl_status tiled_linear_gemm_forward(int64_t T, int64_t K, int64_t n,
                                    const void *x_dev, int64_t ldx,
                                    const void *w_dev, int64_t ldw,
                                    void *y_dev, int64_t ldy, int32_t *err_dev, void *stream);

/* dw[K, n] (bf16, ld lddw) = x[T, K]^T (bf16, ld ldx) . dy[T, n] (bf16, ld lddy). */
tl_status tiled_linear_gemm_dw(int64_t T, int64_t K, int64_t n,
                               const void *x_dev, int64_t ldx,
                               const void *dy_dev, int64_t lddy,
                               void *dw_dev, int64_t lddw, int32_t *err_dev, void *stream);

/* dx[T, K] (fp32, ld lddx) (+)= dy[T, n] (bf16, ld lddy) . w[K, n]^T (bf16,
 * ld ldw); accumulate = 0 overwrites dx, 1 adds to it. */
tl_status tiled_linear_gemm_dx(int64_t T, int64_t K, int64_t n,
                               const void *dy_dev, int64_t lddy,
                               const void *w_dev, int64_t ldw,
                               float *dx_dev, int64_t lddx, int32_t accumulate,
                               int32_t *err_dev, void *stream);

/* dx[T, K] (bf16, ld lddx) = bf16(addend[T, K] + dy[T, n] . w[K, n]^T): the
 * product as tiled_linear_gemm_dx computes it in fp32, plus the fp32 addend
 * (ld ld_add, a multiple of 8 >= K; NULL: no addend), rounded to nearest even
 * once.  A chain's last dX launch per operator writes the previous operator's
 * dY this way (operators in sequence, each tiled as ZeRO-Infinity's
 * "Memory-centric tiling" splits one).  The result equals tiled_linear_gemm_dx
 * with accumulate = 1 into a copy of the addend, then rounded to bf16. */
tl_status tiled_linear_gemm_dx_bf16(int64_t T, int64_t K, int64_t n,
                                    const void *dy_dev, int64_t lddy,
                                    const void *w_dev, int64_t ldw,
                                    const float *addend_dev, int64_t ld_add,
                                    void *dx_dev, int64_t lddx,
                                    int32_t *err_dev, void *stream);

/* Self-test of the kernels' failure path.  Launches the forward GEMM kernel
 * on a 128 x 256 x 64 problem with every operand load withheld and every
 * bounded wait limited to timeout_ns (0 < timeout_ns <= 10 s): the MMA
 * thread's wait for its first shared-memory stage runs out, it sets bit 2 in
 * the int32 at scratch_dev (cleared first, with the tile counter after it),
 * every role stops, the kernel frees its tensor memory and exits -- nothing
 * faults or hangs and the context stays usable.  scratch_dev: device memory,
 * 256-byte aligned, at least 65792 bytes (only the first two int32 are
 * written).  Stream-ordered.
 * Errors: TL_ERR_INVALID, TL_ERR_CUDA. */
tl_status tiled_linear_selftest_timeout(void *scratch_dev, size_t scratch_bytes, int64_t timeout_ns,
                                        void *stream);

/* --- forward without any device allocation --------------------------------
 * The pages describe no counterpart to this entry point.  It exists for
 * callers that cannot allocate device memory at all and so cannot supply the
 * workspace tiled_linear_create needs: for example a plug-in running inside a
 * framework whose allocator owns all of the GPU's memory, or a service that
 * forbids new allocations once it has started.
 *
 * Computes the same Y as tiled_linear_forward for W stored tile-major
 * [N][K][Mi] in pinned host memory, with the same kernel and tile order, so Y
 * is identical.  Its scratch (one weight-tile slot and the kernels' timeout
 * word) is a 32 MiB static device array inside this library, which every GPU
 * that loads the library holds until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *  - Limit: one tile, K*(M/N)*2 bytes, must fit in 32 MiB - 256 bytes; a
 *    larger tile returns TL_ERR_WORKSPACE (split W into more tiles).
 *  - Every copy and GEMM is ordered on `stream`, so copies do not overlap the
 *    GEMMs.
 *  - The first call on each device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *  - All calls share the array, which keeps the last call's contents (the
 *    timeout word is cleared at the start of each call).  Calls whose work
 *    overlaps on the GPU (other streams, other host threads) race on it:
 *    order them.
 *  - status_host: optional (NULL or pinned host int32); receives the kernels'
 *    timeout word once `stream` completes (0 = no timeout).
 * Errors: TL_ERR_INVALID, TL_ERR_NOT_PINNED, TL_ERR_WORKSPACE, TL_ERR_CUDA. */
tl_status tiled_linear_forward_static(int64_t T, int64_t K, int64_t M, int32_t N,
                                      const void *w_host, const void *x_dev, void *y_dev,
                                      int32_t *status_host, void *stream);

/* --- pinned host memory helpers ------------------------------------------ */
/* Page-locked host allocation (cudaHostAlloc, portable); *out = NULL on
 * failure.  Free with tiled_linear_host_free. */
tl_status tiled_linear_host_alloc(size_t bytes, void **out);
tl_status tiled_linear_host_free(void *p);

/* Library version string. */
const char *tiled_linear_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TILED_LINEAR_H */
